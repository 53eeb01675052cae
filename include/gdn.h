/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta-rule verification library.
 *
 * The library runs the Gated DeltaNet recurrence of a hybrid (linear +
 * full attention) model over a speculative verification block and commits
 * the accepted state:
 *
 *     S_n = alpha_n * S_src(n) * (I - beta_n k_n k_n^T) + beta_n v_n k_n^T
 *     o_n = S_n q_n
 *
 * ("TokenSpeed hits 580 tok/s", section "Why Qwen3.5 is hard to serve fast":
 * a fixed d x d state per head, updated per token and queried by q.)
 * S_src(n) is the previous position for a causal chain ("Photon 2.6",
 * section "Speculative verification in a megakernel") and the parent node
 * for a best-first draft tree ("Qwen3.6 27B: From 20 t/s to 184 t/s",
 * DFlash section, steps 3-4).  Every node's state is persisted so that a
 * rejected suffix needs no work ("We got 207 tok/s with Qwen3.5-27B on an
 * RTX 3090", list "Key wins", persist-write kernel), and the accepted node's
 * state is committed into the recurrent-state cache ("Photon 2.6", section
 * "Handling recurrent state").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - The state of one value head is stored TRANSPOSED: H[i][j] = S[j][i],
 *    an fp32 row-major d_k x d_v matrix (i over d_k, j over d_v).
 *  - Value head h reads q/k head h / (Hv / Hk) (contiguous groups).
 *  - No scaling is applied to q; fold any 1/sqrt(d_k) into q beforehand.
 *    q and k are used as given (callers L2-normalise them upstream).
 *  - Every pointer argument is DEVICE memory of the current CUDA device,
 *    allocated and owned by the caller, unless stated otherwise.  The library
 *    allocates nothing and never synchronises: work is enqueued on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream) and the call returns
 *    once it is launched.  It keeps no mutable state between calls, with one
 *    exception: the built-in scratch array of gdn_prefill_chunked_noalloc
 *    (see there for how concurrent calls of that entry point race).
 *  - Profiling ranges: with the environment variable GDN_NVTX set to a value
 *    other than "0" when the library is loaded, every entry point pushes an
 *    NVTX range named after itself for the duration of the host call (so a
 *    timeline tool shows where each launch was issued); unset, the check
 *    costs one branch per call.
 *  - Kernels are launched with programmatic dependent launch allowed: each
 *    kernel starts by waiting until the kernel before it on the stream has
 *    completed and its memory is visible, then lets the next kernel begin
 *    launching.  Stream order is kept for every read and write.  Before that
 *    wait a kernel only issues L2 prefetch hints for lines it will read
 *    (which never change memory).  A kernel of the caller's that follows one
 *    of ours with the same launch attribute must itself wait before reading
 *    our outputs (griddepcontrol.wait), as programmatic launch requires.
 *  - All pointers must be 16-byte aligned; element strides are in elements.
 *  - Host-detected errors return a negative gdn_status before anything is
 *    launched.  Errors that depend on device data (a malformed tree, an
 *    out-of-range accept index or slot) are written to the optional device
 *    word `status` (first error wins; the caller zeroes it) and the affected
 *    sequence is skipped; kernels never trap and never wait on other blocks.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_VERSION 3

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = -1,   /* null pointer, negative or inconsistent size */
  GDN_ERR_UNSUPPORTED = -2,   /* a size outside what the kernels implement */
  GDN_ERR_MISALIGNED = -3,    /* pointer not 16-byte aligned, or stride not a multiple of 4 */
  GDN_ERR_CUDA = -4,          /* the launch itself failed */
  GDN_ERR_BAD_TREE = -5,      /* device: parent[0] != -1 or parent[n] outside [0, n) */
  GDN_ERR_ACCEPT_RANGE = -6,  /* device: accept index outside [0, N) */
  GDN_ERR_SLOT_RANGE = -7,    /* device: slot outside [0, n_slots) */
  GDN_ERR_WORKSPACE = -8,     /* workspace missing or smaller than required */
  GDN_ERR_SCRATCH_LIMIT = -9, /* problem too large for the built-in scratch of the _noalloc call */
  GDN_ERR_TIMEOUT = -10       /* device: a bounded wait on an asynchronous copy or tensor-core
                                 operation expired; that call's outputs are not valid */
} gdn_status;

typedef enum gdn_dtype {
  GDN_F32 = 0,
  GDN_BF16 = 1
} gdn_dtype;

/*
 * Arguments of one verify call (one GDN layer, B sequences, N nodes each).
 *
 *   q, k          [B][N][Hk][dk]  in_dtype (GDN_F32 or GDN_BF16)
 *   v             [B][N][Hv][dv]  in_dtype
 *   alpha, beta   [B][N][Hv]      fp32 gates (decay alpha, write strength beta)
 *   state_cache   recurrent-state cache, READ ONLY here: the state of
 *                 sequence b, head h starts at
 *                 state_cache + slot[b]*cache_slot_stride + h*dk*dv.
 *                 It may be the snapshots buffer itself (index-table
 *                 commit, gdn_commit_index): each sequence's state is read
 *                 before any of its nodes is written
 *   slot          [B] int32 cache slot per sequence; NULL means slot[b] = b
 *   n_slots       number of valid slots (slot[b] is checked against it)
 *   snapshots     [B][N][Hv][dk][dv] fp32 output: S_n of every node.  May be
 *                 NULL (chain or tree): nothing is persisted and the accepted
 *                 state is committed by replay (gdn_replay_accepted)
 *   o             [B][N][Hv][dv] fp32 output
 *   status        optional device int32 error word (see above)
 *   tile_cols, row_warps
 *                 0 = automatic; otherwise the d_v columns owned by one
 *                 thread block (8 or 16) and the warps that split its d_k
 *                 rows (1, or 2 for 16 columns with d_k = 64 or 128).  A
 *                 performance hint: results are identical up to the order
 *                 in which the column sums are added, and a replay commit
 *                 repeats a chain verify bit for bit only with the same
 *                 tile.  GDN_ERR_UNSUPPORTED for any other combination.
 *   max_depth     tree verify only: 0 = no cap; otherwise a sequence whose
 *                 tree has a node deeper than max_depth (the root has depth 1)
 *                 is skipped and GDN_ERR_BAD_TREE is written to `status`.
 *                 Ignored by the chain and replay calls.
 *
 * Supported sizes: dk in {16, 32, 64, 128}; dv a multiple of 16, <= 1024;
 * 1 <= N <= 64; Hv a multiple of Hk; B >= 0 (B = 0 launches nothing).
 */
typedef struct gdn_verify_args {
  const void* q;
  const void* k;
  const void* v;
  const float* alpha;
  const float* beta;
  const float* state_cache;
  const int32_t* slot;
  float* snapshots;
  float* o;
  int32_t* status;
  int64_t cache_slot_stride;
  int32_t n_slots;
  int32_t B;
  int32_t N;
  int32_t Hk;
  int32_t Hv;
  int32_t dk;
  int32_t dv;
  int32_t in_dtype;
  int32_t tile_cols;
  int32_t row_warps;
  int32_t max_depth;
} gdn_verify_args;

/*
 * Causal-chain verification (DFlash block: the last committed token plus the
 * drafts).  Node n starts from node n-1's state; node 0 from the cache.
 * Writes every node's state to `snapshots` (when not NULL) and its output to
 * `o`.
 */
int gdn_verify_chain(const gdn_verify_args* args, void* stream);

/*
 * Tree verification (DDTree block).  parent [B][N] int32 with parent[b][0] = -1
 * (the root, i.e. the last committed token, starts from the cache) and
 * 0 <= parent[b][n] < n otherwise (nodes in topological order).  Node n starts
 * from its parent's state.  depth_out [B][N] int32 (optional, may be NULL)
 * receives each node's depth, root = 1.  A sequence whose parent array breaks
 * the rule, or whose tree is deeper than args->max_depth (when not 0), is
 * skipped and GDN_ERR_BAD_TREE is written to args->status (its depth_out row
 * is still written when the parent array itself is valid).  With
 * args->snapshots == NULL (a block committed by gdn_replay_accepted) the
 * block is verified by one lower-triangular solve per slab instead of the
 * node-by-node walk, and only o (and depth_out) is written; the outputs agree
 * with the walk's up to floating-point rounding.
 */
int gdn_verify_tree(const gdn_verify_args* args, const int32_t* parent, int32_t* depth_out,
                    void* stream);

/*
 * Commit the accepted node of every sequence, for n_layers layers at once:
 *
 *   state_cache[l][slot[b]][h] = snapshots[l][b][accept_idx[b]][h]
 *
 * Layer l of the snapshots starts at snapshots + l*snap_layer_stride and is
 * laid out [B][N][Hv][dk][dv]; layer l of the cache starts at
 * state_cache + l*cache_layer_stride, slot s at + s*cache_slot_stride, head h
 * at + h*dk*dv.  For a chain with accept length L, accept_idx = L - 1.
 * The copy is bit-exact.  An accept index outside [0, N) or a slot outside
 * [0, n_slots) skips that sequence and is reported through `status`.
 * snapshots and state_cache must not overlap, and the slot[] entries of one
 * call must be distinct (two sequences committing into one slot race, and
 * the slot then holds either state).
 */
int gdn_commit_accepted(const float* snapshots, int64_t snap_layer_stride,
                        const int32_t* accept_idx, float* state_cache, int64_t cache_slot_stride,
                        int64_t cache_layer_stride, const int32_t* slot, int32_t n_slots,
                        int32_t B, int32_t N, int32_t Hv, int32_t dk, int32_t dv,
                        int32_t n_layers, int32_t* status, void* stream);

/*
 * Verification and replay from raw projections (input preparation fused into
 * the recurrence kernel).  The same calls as gdn_verify_chain,
 * gdn_verify_tree and gdn_replay_accepted, except that
 *   q, k          are the raw projections: each (node, q/k head) vector is
 *                 L2-normalised in the kernel (a zero vector stays zero);
 *   alpha, beta   hold the gate pre-activations a, b: the kernel uses
 *                 alpha = exp(-softplus(a)) = 1 / (1 + e^a) and
 *                 beta = sigmoid(b) = 1 / (1 + e^-b).
 * These are the maps the block's inputs are defined by (q and k L2-normalised
 * per head, alpha from exp(-softplus), beta from sigmoid).  Results equal the
 * plain calls on the prepared inputs up to floating-point rounding.
 */
int gdn_verify_chain_prep(const gdn_verify_args* args, void* stream);
int gdn_verify_tree_prep(const gdn_verify_args* args, const int32_t* parent, int32_t* depth_out,
                         void* stream);
int gdn_replay_accepted_prep(const gdn_verify_args* args, const int32_t* parent,
                             const int32_t* accept_idx, void* stream);

/*
 * Verification with 16-bit persisted states ("We got 207 tok/s with
 * Qwen3.5-27B on an RTX 3090", list "Key wins": an f16 intermediate cache at
 * half the bandwidth, "at the same tree budget").  The same as
 * gdn_verify_chain / gdn_verify_tree, except that every node's state is
 * written to `snapshots_f16` [B][N][Hv][dk][dv] as IEEE binary16, rounded to
 * nearest even from the fp32 state the kernel forms (args->snapshots is not
 * used).
 *   chain: the recurrence and the outputs o are unchanged; only the
 *          persisted copies are rounded.
 *   tree:  the tree is walked depth level by depth level (the warps of a
 *          block take a level's nodes round robin, in index order).  A node
 *          continues from its parent's exact fp32 state when the warp that
 *          formed the parent takes the node next, or when the parent is one
 *          of the first three nodes of its depth (in index order) that have
 *          children (those stay in shared memory); otherwise it continues
 *          from the parent's binary16 snapshot, as an f16 intermediate cache
 *          does.  The root starts from the fp32 cache.
 */
int gdn_verify_chain_f16(const gdn_verify_args* args, void* snapshots_f16, void* stream);
int gdn_verify_tree_f16(const gdn_verify_args* args, const int32_t* parent, int32_t* depth_out,
                        void* snapshots_f16, void* stream);

/*
 * gdn_commit_accepted for binary16 snapshots: the accepted node's state is
 * widened exactly to fp32 into the cache (so the committed state carries one
 * binary16 rounding per block).  Strides are in elements; same checks and
 * status reporting as gdn_commit_accepted.
 */
int gdn_commit_accepted_f16(const void* snapshots_f16, int64_t snap_layer_stride,
                            const int32_t* accept_idx, float* state_cache,
                            int64_t cache_slot_stride, int64_t cache_layer_stride,
                            const int32_t* slot, int32_t n_slots, int32_t B, int32_t N,
                            int32_t Hv, int32_t dk, int32_t dv, int32_t n_layers,
                            int32_t* status, void* stream);

/*
 * Convolution-history commit ("Photon 2.6", section "Handling recurrent
 * state": the convolution history is committed to the same boundary as the
 * recurrent state).  A short causal convolution before the recurrence keeps,
 * per cache slot and channel, the last W raw inputs (oldest first):
 *
 *   conv_state  slot s, channel c at conv_state + s*state_slot_stride + c*W,
 *               W consecutive elements (in_dtype)
 *   x           [B][N][C] raw inputs of the block's nodes (in_dtype)
 *
 * For every sequence b the history is advanced in place over the accepted
 * path (chain: nodes 0 .. accept_idx[b], parent == NULL; tree: the ancestors
 * of accept_idx[b] from the root, parent [B][N] as in gdn_verify_tree): the
 * new history is the last W elements of [old history, x of the path nodes].
 * The copy is bit-exact.  1 <= W <= 8.  A bad accept index, slot or parent
 * array skips that sequence and is reported through `status`.  The slot[]
 * entries of one call must be distinct: the history is rewritten in place,
 * and two sequences sharing a slot race on it.
 */
int gdn_conv_commit(const void* x, int32_t in_dtype, void* conv_state,
                    int64_t state_slot_stride, const int32_t* slot, int32_t n_slots,
                    const int32_t* parent, const int32_t* accept_idx, int32_t B, int32_t N,
                    int32_t C, int32_t W, int32_t* status, void* stream);

/*
 * Index-table commit ("TokenSpeed hits 580 tok/s", section "How they actually
 * got there": move pointers, not data -- the persisted states form a draft
 * region and a small index table says which one is current).  No state is
 * copied: the slot table is pointed at the accepted node's snapshot,
 *
 *   slot[b] = base_slot + b*N + accept_idx[b]
 *
 * so that a verify call given the snapshots buffer [B][N][Hv][dk][dv] of this
 * block as its state_cache (cache_slot_stride = Hv*dk*dv, n_slots >=
 * base_slot + B*N) starts every sequence from its accepted node; base_slot
 * places the block's region inside a larger slot space.  That verify may
 * write its own snapshots into the same buffer.  An accept index outside
 * [0, N) leaves slot[b] unchanged and is reported through `status`.
 */
int gdn_commit_index(const int32_t* accept_idx, int32_t B, int32_t N, int32_t base_slot,
                     int32_t* slot, int32_t* status, void* stream);

/*
 * Checkpoint-and-replay commit ("Photon 2.6", section "Handling recurrent
 * state": keep the state from before the block and re-run the accepted
 * tokens instead of persisting every node).  For every sequence b the
 * recurrence is run again over the accepted path, starting from the cached
 * state, and the result replaces the cached state in place:
 *
 *   state_cache[slot[b]][h] <- S_{accept_idx[b]} of the block
 *
 * The path is nodes 0 .. accept_idx[b] for a chain (parent == NULL; accept
 * length L = accept_idx + 1) and the ancestors of accept_idx[b] from the root
 * for a tree (parent [B][N] as in gdn_verify_tree).  Uses k, v, alpha, beta,
 * state_cache, slot, n_slots, status and the sizes of `args` (args->q,
 * snapshots and o are not used and may be NULL); here state_cache is read and
 * written.  The state equals snapshots[b][accept_idx[b]] of a verify call on
 * the same inputs up to floating-point rounding.  An accept index outside
 * [0, N), a slot outside [0, n_slots) or a bad parent array skips that
 * sequence and is reported through args->status.  Two sequences must not
 * share a slot.
 */
int gdn_replay_accepted(const gdn_verify_args* args, const int32_t* parent,
                        const int32_t* accept_idx, void* stream);

/*
 * Chunked prefill of one sequence of T tokens: the same recurrence, evaluated
 * chunk by chunk in the WY / UT-transform form on tensor cores.
 *
 *   q, k   [T][Hk][dk]  bf16;  v [T][Hv][dv] bf16
 *   alpha, beta [T][Hv] fp32
 *   state  [Hv][dk][dv] fp32, in: the state before token 0, out: after token T-1
 *   o      [T][Hv][dv] fp32 output
 *   workspace  device scratch of at least gdn_prefill_workspace_bytes(...) bytes,
 *              owned by the caller, contents need not be initialised
 *   status optional device int32 error word (first error wins; the caller
 *          zeroes it): GDN_ERR_TIMEOUT if a bounded wait of the kernel on its
 *          own asynchronous copies or tensor-core work expired.  The kernel
 *          then stops early; the state of the affected heads is written as
 *          NaN, and o is not valid.
 *
 * Supported: dk = dv = 128, chunk = 64, in_dtype = GDN_BF16, T >= 0 (any T;
 * the last chunk may be partial); any other size or dtype returns
 * GDN_ERR_UNSUPPORTED before anything is launched.  GDN_ERR_WORKSPACE if the
 * workspace is NULL or too small.  Two kernels run on `stream`: a parallel
 * pass over (chunk, q/k head) that fills the workspace, then the sequential
 * pass over the chunks of each value head; the workspace may be reused once
 * the call's work has finished on the stream.
 */
size_t gdn_prefill_workspace_bytes(int32_t T, int32_t Hk, int32_t Hv, int32_t dk, int32_t dv,
                                   int32_t chunk);

int gdn_prefill_chunked(const void* q, const void* k, const void* v, int32_t in_dtype,
                        const float* alpha, const float* beta, int32_t T, int32_t Hk, int32_t Hv,
                        int32_t dk, int32_t dv, int32_t chunk, float* state, float* o,
                        void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * gdn_prefill_chunked without a workspace argument, for callers that cannot
 * allocate device memory themselves: for example a plugin whose host engine
 * owns every device allocation and offers it no allocator, or a code path
 * where the implicit synchronisation of cudaMalloc is not acceptable and no
 * buffer was reserved up front.  (The source pages have no counterpart to this
 * call; it is an addition of this library.)
 *
 * The call computes exactly what gdn_prefill_chunked computes, with the same
 * arguments minus `workspace`/`workspace_bytes`; the scratch it needs lives in
 * a device array built into the library of GDN_PREFILL_NOALLOC_SCRATCH_BYTES
 * (16 MiB) per GPU that loads the library, held until the process exits.
 * Limit: ceil(T/64) * Hv * 33280 bytes must fit, i.e. ceil(T/64) * Hv <= 504
 * (T <= 640 tokens at 48 value heads); larger problems return
 * GDN_ERR_SCRATCH_LIMIT without launching anything.  The library allocates
 * nothing here: no cudaMalloc, cudaFree or allocating library routine.
 *
 * Every call looks up the device address of the scratch array on the current
 * device (cudaGetSymbolAddress, a host-side query that is repeated each time
 * so that a reset device or a new context is never handed a stale address).
 * The first such lookup on a device loads the library's device code there;
 * make that first call before any stream capture.  All calls share the one
 * array, which keeps
 * the previous call's contents (nothing in it needs clearing: the first kernel
 * of a call writes every byte the second kernel reads).  Calls that overlap on
 * the GPU -- on different streams, or from different host threads -- race on
 * the shared scratch and must be serialised by the caller.
 */
#define GDN_PREFILL_NOALLOC_SCRATCH_BYTES (16u << 20)

int gdn_prefill_chunked_noalloc(const void* q, const void* k, const void* v, int32_t in_dtype,
                                const float* alpha, const float* beta, int32_t T, int32_t Hk,
                                int32_t Hv, int32_t dk, int32_t dv, int32_t chunk, float* state,
                                float* o, int32_t* status, void* stream);

/* Human-readable name of a gdn_status value (static string, never NULL). */
const char* gdn_status_string(int status);

/* GDN_VERSION of the loaded library. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
