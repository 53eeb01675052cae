// Gated delta-rule oracle: a plain, slow CPU statement of what the verify,
// commit and prefill paths compute.  TEST INFRASTRUCTURE ONLY: it is called by
// tests/, by __graft_entry__.smoke() and by bench.py's CPU baseline, never by
// the library.  It shares no code, header or constant with the CUDA path.
//
// Notation: the gated delta rule of Gated DeltaNet, whose state is a fixed
// d x d matrix updated once per token and read by that token's query
// ("TokenSpeed hits 580 tok/s", section "Why Qwen3.5 is hard to serve fast"):
//
//     S_n = alpha_n * S_src(n) * (I - beta_n k_n k_n^T) + beta_n v_n k_n^T
//     o_n = S_n q_n
//
// S is d_v x d_k.  It is STORED transposed, H[i][j] = S[j][i] with i over d_k
// and j over d_v, row-major: one fp32 d_k x d_v matrix per value head.
// S_src(n) is S_{n-1} for a chain (the cached state for n = 0) and S_parent(n)
// for a tree ("Qwen3.6 27B: From 20 t/s to 184 t/s", DFlash section, steps 3-4:
// a best-first tree verified under its causal / ancestor mask).
//
// The only algebra applied to the definition is distributivity:
//     S (I - beta k k^T) = S - beta (S k) k^T,
// which turns the d^3 matrix product into d^2 work; everything else is the
// equation term by term, in index order.  Arithmetic is in R = double (or
// long double for tiny brute-force cases).  parity pinned by tests/test_oracle_pins.py.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// status codes shared in meaning (not in code) with the library
constexpr int OK = 0;
constexpr int ERR_INVALID_ARG = -1;
constexpr int ERR_BAD_TREE = -5;
constexpr int ERR_ACCEPT_RANGE = -6;
constexpr int ERR_SLOT_RANGE = -7;

// One token / node for one value head.
//   H     [dk][dv]  in: S_src transposed; out: S_n transposed
//   k, q  [dk];  v [dv];  o [dv]
template <typename R>
void gdn_step(R* H, const R* k, const R* v, const R* q, R alpha, R beta, int dk, int dv, R* o,
              std::vector<R>& u) {
  // u = S k, u_j = sum_i S[j][i] k_i
  for (int j = 0; j < dv; ++j) {
    R acc = 0;
    for (int i = 0; i < dk; ++i) acc += H[(int64_t)i * dv + j] * k[i];
    u[j] = acc;
  }
  // S' = alpha * (S - beta * u k^T) + beta * v k^T
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) {
      R s = H[(int64_t)i * dv + j];
      H[(int64_t)i * dv + j] = alpha * (s - beta * u[j] * k[i]) + beta * v[j] * k[i];
    }
  // o = S' q, o_j = sum_i S'[j][i] q_i
  for (int j = 0; j < dv; ++j) {
    R acc = 0;
    for (int i = 0; i < dk; ++i) acc += H[(int64_t)i * dv + j] * q[i];
    o[j] = acc;
  }
}

// parent[0] must be -1 and 0 <= parent[n] < n for n >= 1.  depth(root) = 1.
// A draft tree's depth is capped ("Qwen3.6 27B: From 20 t/s to 184 t/s",
// DFlash section: a best-first tree grown under a budget; the DDTree workload
// caps it at 16): with max_depth > 0, a tree holding a node deeper than the
// cap is rejected after every depth has been filled in.
int tree_depth(const int32_t* parent, int N, int32_t* depth, int max_depth = 0) {
  if (N <= 0) return ERR_INVALID_ARG;
  if (parent[0] != -1) return ERR_BAD_TREE;
  depth[0] = 1;
  for (int n = 1; n < N; ++n) {
    int p = parent[n];
    if (p < 0 || p >= n) return ERR_BAD_TREE;
    depth[n] = depth[p] + 1;
  }
  if (max_depth > 0)
    for (int n = 0; n < N; ++n)
      if (depth[n] > max_depth) return ERR_BAD_TREE;
  return OK;
}

template <typename R>
int verify(const R* q, const R* k, const R* v, const R* alpha, const R* beta, const R* cache,
           int64_t cache_slot_stride, const int32_t* slot, int32_t n_slots, const int32_t* parent,
           int32_t B, int32_t N, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, R* snap, R* o,
           int32_t max_depth) {
  if (B < 0 || N <= 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk != 0)
    return ERR_INVALID_ARG;
  const int G = Hv / Hk;               // value heads per q/k head (contiguous groups)
  const int64_t hs = (int64_t)dk * dv; // one state
  std::vector<R> u(dv);
  std::vector<int32_t> depth(N);
  int status = OK;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent ? parent + (int64_t)b * N : nullptr;
    if (par) {
      int st = tree_depth(par, N, depth.data(), max_depth);
      if (st != OK) { status = st; continue; }
    }
    int sl = slot ? slot[b] : b;
    if (sl < 0 || sl >= n_slots) { status = ERR_SLOT_RANGE; continue; }
    for (int h = 0; h < Hv; ++h) {
      const int hk = h / G;
      const R* S0 = cache + (int64_t)sl * cache_slot_stride + (int64_t)h * hs;
      for (int n = 0; n < N; ++n) {
        int src = par ? par[n] : n - 1;
        const R* from = src < 0 ? S0 : snap + (((int64_t)b * N + src) * Hv + h) * hs;
        R* H = snap + (((int64_t)b * N + n) * Hv + h) * hs;
        std::memcpy(H, from, sizeof(R) * hs);
        const int64_t node = (int64_t)b * N + n;
        gdn_step<R>(H, k + (node * Hk + hk) * dk, v + (node * Hv + h) * dv,
                    q + (node * Hk + hk) * dk, alpha[node * Hv + h], beta[node * Hv + h], dk,
                    dv, o + (node * Hv + h) * dv, u);
      }
    }
  }
  return status;
}

// Checkpoint-and-replay commit ("Photon 2.6", section "Handling recurrent
// state": keep the state from before the block and re-run the accepted tokens
// instead of persisting every node): for every sequence, the recurrence over
// the accepted path (chain: nodes 0 .. accept; tree: the ancestors of accept,
// root first), starting from the cached state, replaces the cached state.
template <typename R>
int replay(const R* k, const R* v, const R* alpha, const R* beta, R* cache,
           int64_t cache_slot_stride, const int32_t* slot, int32_t n_slots, const int32_t* parent,
           const int32_t* accept, int32_t B, int32_t N, int32_t Hk, int32_t Hv, int32_t dk,
           int32_t dv) {
  if (B < 0 || N <= 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk != 0)
    return ERR_INVALID_ARG;
  const int G = Hv / Hk;
  const int64_t hs = (int64_t)dk * dv;
  std::vector<R> u(dv), o(dv), H(hs);
  std::vector<int32_t> depth(N), path;
  int status = OK;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent ? parent + (int64_t)b * N : nullptr;
    if (par) {
      int st = tree_depth(par, N, depth.data());
      if (st != OK) { status = st; continue; }
    }
    const int acc = accept[b];
    if (acc < 0 || acc >= N) { status = ERR_ACCEPT_RANGE; continue; }
    int sl = slot ? slot[b] : b;
    if (sl < 0 || sl >= n_slots) { status = ERR_SLOT_RANGE; continue; }
    // the accepted path, root first
    path.clear();
    if (par) {
      for (int m = acc; m >= 0; m = par[m]) path.insert(path.begin(), m);
    } else {
      for (int m = 0; m <= acc; ++m) path.push_back(m);
    }
    for (int h = 0; h < Hv; ++h) {
      const int hk = h / G;
      R* S = cache + (int64_t)sl * cache_slot_stride + (int64_t)h * hs;
      std::memcpy(H.data(), S, sizeof(R) * hs);
      for (int n : path) {
        const int64_t node = (int64_t)b * N + n;
        const R* kn = k + (node * Hk + hk) * dk;
        // the output is not needed here: k stands in for q
        gdn_step<R>(H.data(), kn, v + (node * Hv + h) * dv, kn, alpha[node * Hv + h],
                    beta[node * Hv + h], dk, dv, o.data(), u);
      }
      std::memcpy(S, H.data(), sizeof(R) * hs);
    }
  }
  return status;
}

}  // namespace

extern "C" {

// Convolution-history commit ("Photon 2.6", section "Handling recurrent
// state": the convolution history is committed to the same boundary as the
// state).  Per cache slot and channel the history holds the last W raw inputs,
// oldest first (state + slot*stride + c*W); for every sequence the new history
// is the last W elements of the old history followed by the channel's inputs
// x[b][n][c] at the nodes of the accepted path (chain: 0 .. accept; tree: the
// ancestors of accept from the root).
int oracle_conv_commit_f64(const double* x, double* state, int64_t slot_stride,
                           const int32_t* slot, int32_t n_slots, const int32_t* parent,
                           const int32_t* accept, int32_t B, int32_t N, int32_t C, int32_t W) {
  if (B < 0 || N <= 0 || C <= 0 || W <= 0) return ERR_INVALID_ARG;
  std::vector<int32_t> depth(N), path;
  std::vector<double> seq;
  int status = OK;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent ? parent + (int64_t)b * N : nullptr;
    if (par) {
      int st = tree_depth(par, N, depth.data());
      if (st != OK) { status = st; continue; }
    }
    const int acc = accept[b];
    if (acc < 0 || acc >= N) { status = ERR_ACCEPT_RANGE; continue; }
    const int sl = slot ? slot[b] : b;
    if (sl < 0 || sl >= n_slots) { status = ERR_SLOT_RANGE; continue; }
    path.clear();
    if (par) {
      for (int m = acc; m >= 0; m = par[m]) path.insert(path.begin(), m);
    } else {
      for (int m = 0; m <= acc; ++m) path.push_back(m);
    }
    for (int c = 0; c < C; ++c) {
      double* h = state + (int64_t)sl * slot_stride + (int64_t)c * W;
      seq.assign(h, h + W);
      for (int n : path) seq.push_back(x[((int64_t)b * N + n) * C + c]);
      for (int w = 0; w < W; ++w) h[w] = seq[seq.size() - W + w];
    }
  }
  return status;
}

// Input preparation of a verify block from raw projections (the maps the
// block's inputs are defined by): q and k L2-normalised per (node, q/k head)
// (a zero vector stays zero), alpha = exp(-softplus(a)), beta = sigmoid(b),
// with softplus(a) = log(1 + e^a) and sigmoid(b) = 1 / (1 + e^-b).
// q, k [rows][d] in place; a, b -> alpha, beta [n] in place.
int oracle_prepare_inputs_f64(double* q, double* k, int64_t rows, int32_t d, double* ab_alpha,
                              double* ab_beta, int64_t n) {
  if (rows < 0 || d <= 0 || n < 0) return ERR_INVALID_ARG;
  for (int64_t r = 0; r < rows; ++r) {
    for (double* x : {q + r * d, k + r * d}) {
      double ss = 0;
      for (int i = 0; i < d; ++i) ss += x[i] * x[i];
      if (ss > 0) {
        const double inv = 1.0 / std::sqrt(ss);
        for (int i = 0; i < d; ++i) x[i] *= inv;
      }
    }
  }
  for (int64_t i = 0; i < n; ++i) {
    const double a = ab_alpha[i], b = ab_beta[i];
    const double softplus = a > 0 ? a + std::log1p(std::exp(-a)) : std::log1p(std::exp(a));
    ab_alpha[i] = std::exp(-softplus);
    ab_beta[i] = 1.0 / (1.0 + std::exp(-b));
  }
  return OK;
}

// Index-table commit ("TokenSpeed hits 580 tok/s", section "How they actually
// got there": move pointers, not data): the accepted node's persisted state is
// made current by pointing the sequence's slot at it in the block's snapshot
// region, slot[b] = base + b*N + accept[b].  A bad accept index leaves the
// slot as it was.
int oracle_commit_index(const int32_t* accept, int32_t B, int32_t N, int32_t base,
                        int32_t* slot) {
  if (B < 0 || N <= 0 || base < 0) return ERR_INVALID_ARG;
  int status = OK;
  for (int b = 0; b < B; ++b) {
    if (accept[b] < 0 || accept[b] >= N) { status = ERR_ACCEPT_RANGE; continue; }
    slot[b] = base + b * N + accept[b];
  }
  return status;
}

// Replay commit, in place on `cache` (same layouts as oracle_verify_f64);
// accept [B] is the accepted node index (chain: accept length - 1).
int oracle_replay_f64(const double* k, const double* v, const double* alpha, const double* beta,
                      double* cache, int64_t cache_slot_stride, const int32_t* slot,
                      int32_t n_slots, const int32_t* parent, const int32_t* accept, int32_t B,
                      int32_t N, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv) {
  return replay<double>(k, v, alpha, beta, cache, cache_slot_stride, slot, n_slots, parent,
                        accept, B, N, Hk, Hv, dk, dv);
}

// Verify one block.  parent == nullptr means a chain (node n continues from
// node n-1, node 0 from the cache).  Layouts:
//   q, k [B][N][Hk][dk]; v [B][N][Hv][dv]; alpha, beta [B][N][Hv]
//   cache: slot s, head h at cache + s*cache_slot_stride + h*dk*dv, [dk][dv]
//   snap [B][N][Hv][dk][dv]; o [B][N][Hv][dv]
// A sequence with an invalid tree or slot is skipped and its error returned;
// max_depth > 0 also rejects a tree deeper than that (root = 1).
int oracle_verify_f64(const double* q, const double* k, const double* v, const double* alpha,
                      const double* beta, const double* cache, int64_t cache_slot_stride,
                      const int32_t* slot, int32_t n_slots, const int32_t* parent, int32_t B,
                      int32_t N, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv, double* snap,
                      double* o, int32_t max_depth) {
  return verify<double>(q, k, v, alpha, beta, cache, cache_slot_stride, slot, n_slots, parent, B,
                        N, Hk, Hv, dk, dv, snap, o, max_depth);
}

int oracle_verify_ld(const long double* q, const long double* k, const long double* v,
                     const long double* alpha, const long double* beta, const long double* cache,
                     int64_t cache_slot_stride, const int32_t* slot, int32_t n_slots,
                     const int32_t* parent, int32_t B, int32_t N, int32_t Hk, int32_t Hv,
                     int32_t dk, int32_t dv, long double* snap, long double* o,
                     int32_t max_depth) {
  return verify<long double>(q, k, v, alpha, beta, cache, cache_slot_stride, slot, n_slots,
                             parent, B, N, Hk, Hv, dk, dv, snap, o, max_depth);
}

// depth[b][n] of each node, root depth 1; returns ERR_BAD_TREE for any
// sequence whose parent array is not topologically ordered from a root at 0,
// or (max_depth > 0) that holds a node deeper than max_depth.
int oracle_tree_depth(const int32_t* parent, int32_t B, int32_t N, int32_t* depth,
                      int32_t max_depth) {
  int status = OK;
  for (int b = 0; b < B; ++b) {
    int st = tree_depth(parent + (int64_t)b * N, N, depth + (int64_t)b * N, max_depth);
    if (st != OK) status = st;
  }
  return status;
}

// Commit the accepted node's state into the cache for every layer:
//   cache[layer][slot[b]][h] = snap[layer][b][accept[b]][h]
// ("Photon 2.6", section "Handling recurrent state": the state at the accepted
// boundary becomes the request's state).  Layer l of snap starts at
// snap + l*snap_layer_stride ([B][N][Hv][dk][dv]); of the cache at
// cache + l*cache_layer_stride with slot stride cache_slot_stride.
int oracle_commit_f64(const double* snap, int64_t snap_layer_stride, const int32_t* accept,
                      double* cache, int64_t cache_slot_stride, int64_t cache_layer_stride,
                      const int32_t* slot, int32_t n_slots, int32_t B, int32_t N, int32_t Hv,
                      int32_t dk, int32_t dv, int32_t n_layers) {
  const int64_t hs = (int64_t)dk * dv;
  int status = OK;
  for (int l = 0; l < n_layers; ++l)
    for (int b = 0; b < B; ++b) {
      int a = accept[b];
      int sl = slot ? slot[b] : b;
      if (a < 0 || a >= N) { status = ERR_ACCEPT_RANGE; continue; }
      if (sl < 0 || sl >= n_slots) { status = ERR_SLOT_RANGE; continue; }
      for (int h = 0; h < Hv; ++h) {
        const double* from = snap + l * snap_layer_stride + (((int64_t)b * N + a) * Hv + h) * hs;
        double* to = cache + l * cache_layer_stride + sl * cache_slot_stride + (int64_t)h * hs;
        for (int64_t e = 0; e < hs; ++e) to[e] = from[e];
      }
    }
  return status;
}

// Prefill: the same recurrence run token by token over one sequence (the
// step form; the chunked kernel must reach the same result).
//   q, k [T][Hk][dk]; v [T][Hv][dv]; alpha, beta [T][Hv]
//   state [Hv][dk][dv] in/out; o [T][Hv][dv]
// heads [h0, h0+nh) only, so tests can sample heads of a large problem.
int oracle_prefill_step_f64(const double* q, const double* k, const double* v,
                            const double* alpha, const double* beta, int32_t T, int32_t Hk,
                            int32_t Hv, int32_t dk, int32_t dv, int32_t h0, int32_t nh,
                            double* state, double* o) {
  if (T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || h0 < 0 || nh < 0 || h0 + nh > Hv)
    return ERR_INVALID_ARG;
  const int G = Hv / Hk;
  const int64_t hs = (int64_t)dk * dv;
  std::vector<double> u(dv);
  for (int h = h0; h < h0 + nh; ++h) {
    double* H = state + (int64_t)h * hs;
    for (int t = 0; t < T; ++t) {
      gdn_step<double>(H, k + ((int64_t)t * Hk + h / G) * dk, v + ((int64_t)t * Hv + h) * dv,
                       q + ((int64_t)t * Hk + h / G) * dk, alpha[(int64_t)t * Hv + h],
                       beta[(int64_t)t * Hv + h], dk, dv, o + ((int64_t)t * Hv + h) * dv, u);
    }
  }
  return OK;
}

}  // extern "C"
