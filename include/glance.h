/*
 * glance.h -- C ABI of the GLANCE verify-round library (sm_103a).
 *
 * One speculative-decoding round of GLANCE ("Vision Is Not Overhead: One-Pass
 * Block Drafting for Lossless Speculative Decoding in Vision-Language Models",
 * arXiv 2609.00355) has four data-parallel steps, one entry point each:
 *
 *   glance_build_tree      draft marginals q_1..q_L -> top-N candidate tree,
 *                          packed (Assumption 1, Definition 1, Section 4.2)
 *   glance_tree_attention  ancestor-masked GQA attention of the packed rows
 *                          against the cached prefix (Definition 1)
 *   glance_lmhead_argmax   LM head of the verified rows with per-row greedy
 *                          argmax and top-2 gap (Section 3.1; Appendix B.1)
 *   glance_accept_commit   acceptance walk A(S), KV commit, bonus root
 *                          (Definition 1; Appendix B.1 proof of Theorem 1)
 *
 * Each step also has a batched form (glance_*_batched) that runs the rounds
 * of B <= 16 independent requests in one launch: same L, V, N and head
 * geometry, but each request has its own draft logits, root, prefix length T
 * (ragged) and KV caches. The LM head needs no batched form: the B requests'
 * rows are stacked into one h of M = B (N + 1) <= 512 rows.
 *
 * Beyond the round itself: the root entropy fused into the LM head
 * (glance_lmhead_argmax_entropy), a sampled rather than greedy verify
 * (glance_lmhead_sample), the tie-aware gate on the walk
 * (glance_accept_commit_gated), one tree budget shared by a batch
 * (glance_build_tree_shared), and the target's dense layers around tree
 * attention (glance_dense_qkv, glance_dense_residual, glance_dense_swiglu,
 * glance_row_sumsq).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Memory: every array argument is a DEVICE pointer unless its comment says
 *   host. The caller owns all memory; the library allocates and frees nothing.
 *   Scratch space is a caller-provided device workspace whose size the
 *   matching *_workspace_bytes() call returns. A workspace must be zero-filled
 *   before its first use; every call leaves the counters it uses at zero, so
 *   the same workspace can be reused by later calls on the same stream. Two
 *   calls that may run at the same time need distinct workspaces.
 * - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream). Every call only enqueues work on that stream and returns; no call
 *   synchronises with the device, so rounds can be captured in a CUDA graph.
 * - Errors: argument errors are found on the host before anything is
 *   launched and are returned as a status; glance_last_error() then describes
 *   them (thread-local text). A failed launch returns GLANCE_ERR_CUDA. Errors
 *   that only the device can see (non-finite draft logits, a prefix length
 *   that leaves no room for the tree rows, a pipeline wait that ran out) set a
 *   device status word and the kernel returns early; glance_get_status()
 *   copies the words out in stream order, glance_device_status() reads them
 *   after a device synchronisation.
 * - Packed tree layout (rows = N + 1; row 0 is the pending root b): rows are
 *   in canonical order: root, then by depth ascending, then by parent row
 *   ascending, then by the node's rank in its offset's candidate list
 *   ascending. Every parent row precedes its children.
 * - KV cache layout, per layer: K and V are separate arrays of
 *   [n_kv_heads][t_cap][head_dim] elements (strides in glance_kv). Slots
 *   0..T-1 hold the committed prefix; the verify pass writes the tree rows'
 *   K/V to slots T..T+N (row r at slot T + r) before attention reads them.
 *   T lives in device memory (*t_len) so that a captured round can be
 *   replayed: kernels read it there and glance_accept_commit advances it.
 */
#ifndef GLANCE_H
#define GLANCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GLANCE_OK = 0,
  GLANCE_ERR_INVALID_ARG = 1, /* null pointer, size out of range, misaligned */
  GLANCE_ERR_UNSUPPORTED = 2, /* a valid shape this build has no kernel for */
  GLANCE_ERR_CAPACITY = 3,    /* workspace too small */
  GLANCE_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  GLANCE_ERR_DEVICE = 5       /* the device status word is set */
} glance_status;

typedef enum { GLANCE_F32 = 0, GLANCE_BF16 = 1 } glance_dtype;

/* Device status word values (glance_device_status). */
#define GLANCE_DEV_OK 0
#define GLANCE_DEV_NONFINITE_LOGITS 1 /* a draft logit row held NaN or +-inf */
#define GLANCE_DEV_TREE_CAPACITY 2    /* the rows' K/V slots do not fit: T + rows > t_cap */
#define GLANCE_DEV_BAD_TREE 3         /* a tree array was inconsistent */
#define GLANCE_DEV_PIPELINE_TIMEOUT 4 /* a pipeline wait ran out of time (2 s) */
#define GLANCE_DEV_OUT_OF_BOUNDS 5    /* bounds-checked build (GLANCE_CHECK) only: a computed
                                        index fell outside its buffer; the access was skipped */

/* A packed candidate tree: device arrays with N + 1 rows, caller-allocated. */
typedef struct {
  int32_t n;          /* N, the budget: non-root nodes (1 <= N <= 255) */
  int32_t L;          /* maximum depth = number of draft offsets (1..16) */
  int32_t mask_words; /* ceil((N+1)/64), 1..4 */
  int32_t* token;     /* [N+1] token id of each row; row 0 = root b */
  int32_t* parent;    /* [N+1] parent row; -1 at the root */
  int32_t* depth;     /* [N+1] 0 at the root */
  int32_t* pos_id;    /* [N+1] position id = T + depth */
  float* score;       /* [N+1] log plug-in score sum_j log q_j(y_j); 0 at root */
  uint64_t* anc;      /* [N+1][mask_words]; bit k of row i (word k/64, bit
                         k%64) is set iff row k is row i, the root, or an
                         ancestor of row i */
} glance_tree;

/* One layer's KV cache view. */
typedef struct {
  void* k;             /* device [n_kv_heads][t_cap][head_dim] elements */
  void* v;             /* same shape as k */
  glance_dtype dtype;  /* GLANCE_BF16 (head_dim 128) or GLANCE_F32 (any
                          head_dim that is a multiple of 32, <= 128) */
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t t_cap;       /* slots per head */
  int64_t head_stride; /* elements between heads (>= t_cap * row_stride) */
  int64_t row_stride;  /* elements between slots (>= head_dim) */
  int32_t* t_len;      /* device int32: T, the committed prefix length */
} glance_kv;

/* ------------------------------------------------------------------ build */

/* Workspace bytes for glance_build_tree with these sizes (0 on bad sizes). */
size_t glance_build_tree_workspace_bytes(int L, int V, int N);

/*
 * Draft-to-tree (Assumption 1; Definition 1; Section 4.2 "the builder keeps
 * the prefixes of highest plug-in score").
 *
 * draft_logits: [L][V] row-major, dtype F32 or BF16; q_j = softmax(row j).
 * For each offset j the kernel forms log q_j = x_j - logsumexp(x_j) and the
 * K = min(N, V) best tokens by (logit desc, token id asc). It then keeps the N
 * strings of highest plug-in score sum_{j<=d} log q_j(y_j) (fp32, summed in
 * order j = 1..d), nodes ordered by (score desc, depth asc, rank vector
 * lexicographic asc), and writes them in canonical packed order.
 * root_token: device int32, the pending root b (row 0's token).
 * t_len: device int32, T (pos_id = T + depth).
 * tree: host struct holding device arrays sized for N+1 rows; tree->n must be
 * N, tree->L must be L and tree->mask_words must be ceil((N+1)/64).
 * Limits: 1 <= L <= 16, 2 <= V <= 262144, 1 <= N <= 255,
 * N <= number of strings of length <= L over V tokens, and
 * ceil(V / 8192) * min(N, V) <= 8192 (the per-row candidate merge).
 */
glance_status glance_build_tree(const void* draft_logits, glance_dtype dtype, int L, int V,
                                int N, const int32_t* root_token, const int32_t* t_len,
                                const glance_tree* tree, void* workspace,
                                size_t workspace_bytes, void* stream);

/* -------------------------------------------------------------- attention */

/* Workspace bytes for glance_tree_attention (0 on bad sizes). */
size_t glance_tree_attention_workspace_bytes(int n_rows, int n_q_heads, const glance_kv* kv);

/*
 * Ancestor-masked tree attention of one layer (Definition 1: each packed row
 * of a depth-d node sees the cached prefix, the root and its own ancestors,
 * so it yields the same row as the unpacked sequence x . b . y_{1:d}).
 *
 * q:   [N+1][n_q_heads][head_dim] (dtype of kv), rotary position already
 *      applied by the caller.
 * kv:  the layer's cache; prefix at slots 0..T-1, tree rows at T..T+N.
 * For q head h the kv head is h / (n_q_heads / n_kv_heads). Row i attends to
 * prefix slots 0..T-1 and tree slots T + k for every k with anc bit (i, k),
 * with scores (q . k) * scale and a softmax over exactly those keys.
 * out: [N+1][n_q_heads][head_dim], same dtype (bf16 rounded to nearest even).
 * Supported: BF16 with head_dim 128, n_q_heads / n_kv_heads in {1,2,4,8},
 * N + 1 <= 256; F32 with head_dim a multiple of 32 up to 128.
 * The BF16 call is a programmatic dependent of the previous kernel in the
 * stream: it may read T and the cache prefix (slots < T) before that kernel
 * has finished, when that kernel lets dependents start early (this library's
 * attention and dense calls do; they never write T or the prefix). q and the
 * tree rows' K/V are read only after it has finished. A T that changes in
 * between sets device status 3 and the call writes nothing.
 */
glance_status glance_tree_attention(const void* q, int n_q_heads, const glance_kv* kv,
                                    const glance_tree* tree, float scale, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Check of the bf16 attention kernel's failure path (no counterpart in the
 * paper; for tests and health checks). Runs glance_tree_attention with every
 * pipeline wait limited to wait_ns nanoseconds (1 us .. 2 s; the normal call
 * uses 2 s) and with the copy of each CTA's last key tile of V never made,
 * unless that tile was fetched before the call's dependency wait, so that the
 * MMA warp's wait for it runs out. That CTA then sets device status 4
 * (GLANCE_DEV_PIPELINE_TIMEOUT), lets its other roles leave, waits for its
 * copies in flight, frees its tensor memory and returns; the launch ends
 * normally and the context stays usable. out is left undefined. Arguments as
 * for glance_tree_attention, BF16 only.
 */
glance_status glance_tree_attention_timeout_check(const void* q, int n_q_heads,
                                                  const glance_kv* kv, const glance_tree* tree,
                                                  float scale, void* out, void* workspace,
                                                  size_t workspace_bytes,
                                                  unsigned long long wait_ns, void* stream);

/* ----------------------------------------------------------------- LM head */

/* Workspace bytes for glance_lmhead_argmax (0 on bad sizes). */
size_t glance_lmhead_argmax_workspace_bytes(int M, int d, int V, glance_dtype dtype);

/*
 * LM head with fused greedy argmax and top-2 gap (Section 3.1: greedy emits
 * argmax_w p(w | prefix); Appendix B.1: gamma = l_(1) - l_(2)).
 *
 * h: [M][d] row-major; W: [d][V] row-major (V contiguous); both dtype.
 * logits[i][v] = sum_k h[i][k] * W[k][v], accumulated in fp32; they are
 * never written out. argmax[i] (int32) is the lowest token id among equal
 * maxima; gap[i] = max logit - largest logit of any other token (0 on an
 * exact tie); maxlogit[i] the max logit (nullable).
 * Supported: BF16 with d % 64 == 0, V % 8 == 0, 1 <= M <= 512; F32 with any
 * d, V and M <= 512. BF16 runs as one launch that streams W once for all M
 * rows (M > 128: all row blocks of a vocabulary tile share each W stage).
 */
glance_status glance_lmhead_argmax(const void* h, const void* W, glance_dtype dtype, int M,
                                   int d, int V, int32_t* argmax, float* gap,
                                   float* maxlogit, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * glance_lmhead_argmax plus each row's next-token entropy (Section 6 and
 * Equation 2: the law that sets the accepted length is keyed on the target's
 * next-token entropy H at the round root; Proposition 1 in Appendix B). For
 * row i, entropy[i] = -sum_v p_v ln p_v in nats with p = softmax(logits[i]),
 * accumulated in the same pass over the logit tiles as the argmax (fp32 sums
 * relative to the running maximum), so row 0 of each request's packed tree
 * gives its round's root entropy. BF16 only (F32 returns
 * GLANCE_ERR_UNSUPPORTED); same workspace size and limits as
 * glance_lmhead_argmax. entropy: device float [M], required.
 */
glance_status glance_lmhead_argmax_entropy(const void* h, const void* W, glance_dtype dtype, int M,
                                           int d, int V, int32_t* argmax, float* gap,
                                           float* maxlogit, float* entropy, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * Sampling-mode LM head (Section 5.4: under sampling the committed token is a
 * draw from the target's own verified row, so the walk of Definition 1 runs
 * unchanged on these tokens and preserves the target's distribution).
 * tokens[i] = argmax_v (l_iv * inv_temperature + g_iv), a draw from
 * softmax(l_i / T); g_iv = -ln(-ln u) with u from Philox4x32-10 (Salmon et
 * al., SC 2011): counter (v / 4, position[i], seq ? seq[i] : 0, 0), key (seed
 * low 32 bits, seed high 32 bits), output word v % 4, u = (top 23 bits of the
 * word + 1/2) / 2^23. position[i] (device int32 [M], required) is the
 * absolute sequence position of the token row i predicts (a packed row's
 * pos_id + 1); seq (device int32 [M], nullable) separates streams, e.g. the
 * requests of a batch. Noise keyed by position makes tree rounds reproduce
 * sampled autoregression of the same seed token for token. gap[i] is the
 * top-2 margin of the perturbed values. F32 or BF16, same limits and
 * workspace as glance_lmhead_argmax; inv_temperature must be finite and > 0.
 */
glance_status glance_lmhead_sample(const void* h, const void* W, glance_dtype dtype, int M, int d,
                                   int V, float inv_temperature, uint64_t seed,
                                   const int32_t* position, const int32_t* seq, int32_t* tokens,
                                   float* gap, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * LM head that allocates nothing and takes no workspace. The paper has no
 * counterpart: this is a convenience of the library. It is for callers that
 * must not allocate device memory or pass scratch space on this path, for
 * example code that runs while a stream is captured in a mode that forbids
 * cudaMalloc, or an engine that has reserved all device memory for its own
 * pool and has none to lend.
 *
 * Same results, arguments and outputs as glance_lmhead_argmax, BF16 only
 * (d % 64 == 0, V % 8 == 0, 1 <= M <= 512; anything else is rejected with an
 * error, F32 with GLANCE_ERR_UNSUPPORTED). Cost: the rows run in blocks of
 * 128, one launch per block, and each launch streams all of W, so a call with
 * M > 128 reads W ceil(M / 128) times (about 5 GB at M = 512, V = 151936,
 * d = 4096, against 1.25 GB for glance_lmhead_argmax). Its scratch (a merge ticket and the
 * partial results of at most 160 CTAs, 240 KB in total) is a file-scope device
 * array of the library, held by every GPU that loads the library until the
 * process exits. Each call clears the ticket with cudaMemsetAsync on `stream`;
 * no call makes cudaMalloc, cudaFree or any other allocating call. The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current: make that first call before any stream capture.
 * The address is kept with the device's context and looked up again (the
 * same set-up) on the first call after that context changes, e.g. after
 * cudaDeviceReset.
 * All calls on a device share the array, which keeps the last call's
 * contents, so calls that may overlap on the GPU (other streams or threads)
 * race with each other: serialise them.
 */
glance_status glance_lmhead_argmax_noalloc(const void* h, const void* W, glance_dtype dtype,
                                           int M, int d, int V, int32_t* argmax, float* gap,
                                           float* maxlogit, void* stream);

/*
 * W as the LM head streams it, for glance_lmhead_argmax_packed: the same
 * computation as glance_lmhead_argmax (Section 3.1; Appendix B.1), with W
 * read in one contiguous 32 KB copy per pipeline stage instead of 64-column
 * boxes of rows 303 KB apart. W is a model constant: pack it once.
 *
 * glance_lmhead_packed_w_bytes: the size of the packed buffer for a BF16 W
 * [d][V] (ceil(V / 256) * (d / 64) * 32 KB), or 0 unless d % 64 == 0,
 * d >= 64, V % 8 == 0.
 *
 * glance_lmhead_pack_w: W (device BF16 [d][V], row-major) -> W_packed (device,
 * caller-owned, packed_bytes >= the size above; both 16-byte aligned), on
 * `stream`. Layout: block (t, kb), t the 256-column tile and kb the 64-row
 * slice of d, at byte (t * (d / 64) + kb) * 32768; inside it four 8 KB boxes
 * of 64 columns; row r of a box at r * 128 bytes, its 16-byte chunk c
 * (columns 8c..8c+7) at chunk position c XOR (r mod 8); columns >= V zero.
 * Errors: null pointers, unsupported shapes, a short buffer, misalignment.
 *
 * glance_lmhead_argmax_packed: glance_lmhead_argmax (greedy) with W given
 * packed; BF16, 1 <= M <= 128, the same workspace
 * (glance_lmhead_argmax_workspace_bytes) and outputs, bit-identical results.
 */
size_t glance_lmhead_packed_w_bytes(int d, int V);
glance_status glance_lmhead_pack_w(const void* W, int d, int V, void* W_packed, size_t packed_bytes,
                                   void* stream);
glance_status glance_lmhead_argmax_packed(const void* h, const void* W_packed, int M, int d, int V,
                                          int32_t* argmax, float* gap, float* maxlogit, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------ commit */

/* Workspace bytes for glance_accept_commit. */
size_t glance_accept_commit_workspace_bytes(int n_layers);

/*
 * Acceptance walk and commit (Definition 1; Appendix B.1 proof of Theorem 1).
 *
 * argmax: [N+1] the target's greedy token of every packed row.
 * Walk: u = root; while depth(u) < L and u has a child whose token equals
 * argmax[u], move to that child. a = A(S) = depth of the last row; the
 * accepted tokens are the tokens of the path rows 1..a; new_root = argmax of
 * the last row.
 * Commit, for every layer in layers[0..n_layers-1] (host array of views): the
 * K and V of path rows path_0 = 0, ..., path_a move from slots T + path_i to
 * slots T + i (all sources are read before any slot is written), then
 * *t_len += a + 1 (every layer must share the same t_len pointer).
 * Outputs (device): n_accepted (int32), accepted_tok ([L] int32, first a
 * valid), new_root (int32; may alias the next round's root_token).
 * Limits: 1 <= n_layers <= 128.
 */
glance_status glance_accept_commit(const glance_tree* tree, const int32_t* argmax,
                                   const glance_kv* layers, int n_layers, int32_t* n_accepted,
                                   int32_t* accepted_tok, int32_t* new_root, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * Tree rows' K/V into the caches (Definition 1: the verify pass evaluates the
 * packed rows in one pass with the prefix, so their K/V sit at slots
 * T..T+N of each layer's cache while tree attention runs; row r at T + r).
 * For callers whose rows' K/V come from elsewhere (another device, the host):
 * one launch writes every layer's rows.
 * src: device, [n_layers][2][n_kv_heads][rows][head_dim] elements of the
 * layers' dtype (K before V), contiguous, 16-byte aligned.
 * layers: host array [n_layers] of views with the same t_len, dtype and
 * geometry; T = *t_len is read on the device. If T + rows > t_cap the call
 * sets device status 2 and writes nothing. Limits: 1 <= n_layers <= 128,
 * 1 <= rows <= 256, rows and strides multiples of 16 bytes.
 */
glance_status glance_kv_write_rows(const void* src, const glance_kv* layers, int n_layers, int rows,
                                   void* stream);

/* ----------------------------------------------------------------- batched */

/*
 * B requests in one launch per step (1 <= B <= 16). These calls compute, for
 * every request r, exactly what the single-request call computes on request
 * r's arguments; the paper defines one round per request (Definition 1), and
 * a batch is B independent rounds.
 *
 * Layout: per-request device arrays are stacked along a leading B axis
 * (draft_logits [B][L][V], root_token [B], q and out [B][N+1][n_q_heads][128],
 * argmax [B][N+1], n_accepted [B], accepted_tok [B][L], new_root [B]).
 * Per-request descriptors are HOST arrays: trees [B] (all sized for the same
 * N and L), and the KV views described at each call.
 */

/* Workspace bytes for glance_build_tree_batched (0 on bad sizes). */
size_t glance_build_tree_batched_workspace_bytes(int B, int L, int V, int N);

/*
 * glance_build_tree for B requests. t_len: device int32 [B], request r's T.
 * Same limits as glance_build_tree.
 */
glance_status glance_build_tree_batched(const void* draft_logits, glance_dtype dtype, int B,
                                        int L, int V, int N, const int32_t* root_token,
                                        const int32_t* t_len, const glance_tree* trees,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for glance_build_tree_shared (0 on bad sizes). */
size_t glance_build_tree_shared_workspace_bytes(int B, int L, int V, int N_max);

/*
 * Trees of B rounds under one shared verifier budget (Appendix B.5,
 * Propositions 4-6: the allocation maximising total expected committed length
 * is global best-first over all rounds' nodes, the law keying each round's
 * node masses by its root entropy, Equation 5). Node s of request r has mass
 * w_r * pi_hat_r(s); the N_total nodes of highest mass are kept, at most N_max
 * per request (its tree capacity). w_r = p_m (1 - p_m^L) with logit p_m =
 * law_b0 - law_b1 * H_r (Equation 2, the geometric mean truncated at L) when
 * root_entropy (device float [B], e.g. row 0 of the previous round's
 * glance_lmhead_argmax_entropy) is given, else 1. Request r keeps the best
 * n_r = n_active[r] (device int32 [B]) nodes of its own best-first order,
 * packed canonically in rows 1..n_r; rows n_r+1..N_max are inactive (token
 * -1, parent -1, depth 0, pos_id T, score -inf, ancestor mask = the row
 * itself) and the walk never reaches them. Equal masses go to the lower
 * request. Trees are sized for N = N_max; other arguments and limits as
 * glance_build_tree_batched. Two launches (search, then allocate and pack).
 */
glance_status glance_build_tree_shared(const void* draft_logits, glance_dtype dtype, int B, int L,
                                       int V, int N_max, int N_total, const int32_t* root_token,
                                       const int32_t* t_len, const float* root_entropy,
                                       float law_b0, float law_b1, const glance_tree* trees,
                                       int32_t* n_active, void* workspace, size_t workspace_bytes,
                                       void* stream);

/* Workspace bytes for glance_tree_attention_batched (0 on bad sizes); the
 * split of the key range over CTAs depends on every request's t_cap, so pass
 * the same kv array as to the call. */
size_t glance_tree_attention_batched_workspace_bytes(int B, int n_rows, int n_q_heads,
                                                     const glance_kv* kv);

/*
 * glance_tree_attention for B requests of one layer. kv: host array [B],
 * request r's cache of this layer (its own k, v, t_cap, strides and t_len;
 * n_kv_heads and head_dim shared). BF16 with head_dim 128 only (F32 returns
 * GLANCE_ERR_UNSUPPORTED). The key range of request r is split over about
 * t_cap_r / (work per CTA) CTAs; the split that finishes a (request, kv head,
 * query tile) last merges it, so no CTA waits for another.
 */
glance_status glance_tree_attention_batched(const void* q, int n_q_heads, const glance_kv* kv,
                                            const glance_tree* trees, int B, float scale,
                                            void* out, void* workspace, size_t workspace_bytes,
                                            void* stream);

/* Workspace bytes for glance_accept_commit_batched (0 on bad sizes). */
size_t glance_accept_commit_batched_workspace_bytes(int B, int n_layers);

/*
 * glance_accept_commit for B requests. layers: host array [B][n_layers],
 * request r's views at layers[r * n_layers + l]; all layers of a request share
 * its geometry and t_len, and no two requests share a t_len. Limits:
 * 1 <= n_layers <= 128, B * n_layers <= 1024.
 */
glance_status glance_accept_commit_batched(const glance_tree* trees, int B,
                                           const int32_t* argmax, const glance_kv* layers,
                                           int n_layers, int32_t* n_accepted,
                                           int32_t* accepted_tok, int32_t* new_root,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream);

/*
 * glance_accept_commit with the tie-aware gate (Section 4.2; the end of the
 * proof of Theorem 1 in Appendix B.1): gap: device float [N+1] (batched:
 * [B][N+1]), the rows' top-2 logit margins from the LM head. The walk stops
 * at the first visited row whose margin is below gate_threshold, a near-tie
 * where reduced precision may reorder the target's two best tokens; the round
 * commits the path up to that row and sets gated (device int32, [B] when
 * batched) to 1, meaning that row's packed argmax (reported as new_root) is
 * not trusted and the caller recomputes the target's own token there.
 * Otherwise gated = 0 and the result equals glance_accept_commit's. The pages
 * print no threshold value; a threshold <= 0 never gates. Same workspace as
 * the ungated calls.
 */
glance_status glance_accept_commit_gated(const glance_tree* tree, const int32_t* argmax,
                                         const float* gap, float gate_threshold,
                                         const glance_kv* layers, int n_layers,
                                         int32_t* n_accepted, int32_t* accepted_tok,
                                         int32_t* new_root, int32_t* gated, void* workspace,
                                         size_t workspace_bytes, void* stream);

glance_status glance_accept_commit_gated_batched(const glance_tree* trees, int B,
                                                 const int32_t* argmax, const float* gap,
                                                 float gate_threshold, const glance_kv* layers,
                                                 int n_layers, int32_t* n_accepted,
                                                 int32_t* accepted_tok, int32_t* new_root,
                                                 int32_t* gated, void* workspace,
                                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ dense layers */

/*
 * The target's dense verify layers around tree attention, at the verify width
 * (1 <= M <= 128 packed rows), for a Qwen3-shaped pre-norm decoder layer. The
 * pages run the frozen target once over the packed rows (Definition 1,
 * Section 4.2) and its forward is most of a round's cost (Table 11); they do
 * not describe the layer, so this one reads it as:
 *   x -> RMSNorm -> [q | k | v] = . W_qkv -> per-head RMSNorm of q and k
 *   (optional) -> rotate-half RoPE -> tree attention -> x + . W_o = x'
 *   x' -> RMSNorm -> SiLU(. W_gate) * (. W_up) -> x' + . W_down.
 * All bf16 row-major, W as [in][out] (out contiguous), fp32 accumulation.
 * An RMSNorm weight g is folded into the next projection by the caller
 * (W <- diag(g) W); the 1 / rms row scale is applied to the product. A call
 * that normalises its input takes the input rows' sums of squares as
 * in_sumsq [n_sumsq][M] partial sums (row scale 1 / sqrt(sum_t in_sumsq[t][row]
 * / d + eps); null: no input norm). glance_dense_residual writes them for its
 * own output (out_sumsq [N / 256][M], nullable), so a layer passes them on;
 * glance_row_sumsq makes them for rows from anywhere else. Each projection is
 * one launch of thread-block clusters that split K (no workspace); it is a
 * programmatic dependent of the previous kernel in the stream. The output must
 * not overlap the input x (other CTAs may still be reading it).
 */

/* sumsq[i] = sum_k x[i][k]^2 (device float [M]; the [1][M] in_sumsq of a
 * following call); x bf16 [M][d], d % 8 == 0. */
glance_status glance_row_sumsq(const void* x, int M, int d, float* sumsq, void* stream);

/*
 * QKV projection of h [M][d] with W_qkv [d][(Hq + 2 Hkv) * 128] (q heads,
 * then k heads, then v heads), rows RMS-scaled from in_sumsq; q and k each
 * get a per-head RMSNorm (weights q_norm / k_norm [128], nullable = none,
 * eps) and rotate-half RoPE at pos_id [M] with base rope_theta (dims j and
 * j + 64 rotate by pos * theta^(-2j/128)). q goes to q_out [M][Hq][128]; k
 * and v go to the cache kv (bf16, head_dim 128) at slots T + row
 * (T = *kv->t_len; if T + M > t_cap, device status 2 and no cache row is
 * written). Hq, Hkv even, Hq % Hkv == 0, d % 64 == 0.
 */
glance_status glance_dense_qkv(const void* h, const void* W_qkv, int M, int d, int n_q_heads,
                               const float* in_sumsq, int n_sumsq, const float* q_norm,
                               const float* k_norm, float eps, const int32_t* pos_id,
                               float rope_theta, void* q_out, const glance_kv* kv, void* stream);

/* out [M][N] = residual [M][N] + x [M][K] W [K][N] (out may alias residual,
 * not x), and out_sumsq [N / 256][M] (nullable) = per 256-column tile, the
 * sums of squares of the rows' stored bf16 outputs; K % 64 == 0,
 * N % 256 == 0. The output and down projections. */
glance_status glance_dense_residual(const void* x, const void* W, int M, int K, int N,
                                    const void* residual, void* out, float* out_sumsq,
                                    void* stream);

/* act [M][inter] = SiLU(r h W_gate) * (r h W_up), r the row's RMS scale from
 * in_sumsq (null: 1); W_gate, W_up [d][inter], inter % 128 == 0,
 * d % 64 == 0. */
glance_status glance_dense_swiglu(const void* h, const void* W_gate, const void* W_up, int M,
                                  int d, int inter, const float* in_sumsq, int n_sumsq, float eps,
                                  void* act, void* stream);

/* ------------------------------------------------------------------ status */

/* Text of the last host-side error on this thread ("" if none). */
const char* glance_last_error(void);

/* Name of a status value. */
const char* glance_status_string(glance_status s);

/* Synchronises the current device, then stores the device status word (one
 * of GLANCE_DEV_*; the first error since the last reset wins) in *code_out
 * (host pointer). Returns GLANCE_ERR_DEVICE if it is non-zero. */
glance_status glance_device_status(int32_t* code_out);

/* Clears the device status word of the current device (synchronous). */
glance_status glance_reset_device_status(void);

/* Number of int32 words glance_get_status writes. */
#define GLANCE_STATUS_WORDS 6

/*
 * Stream-ordered read of the device status words: enqueues on `stream`, after
 * the work already there, copies of the status word of each kernel family
 * into status_out[1..5] (tree build, tree attention, LM head, walk + commit,
 * dense layers) and a one-thread kernel that stores the first non-zero of
 * them in status_out[0] (0 if none). status_out: GLANCE_STATUS_WORDS int32,
 * device memory or pinned / managed host memory (the caller reads it once
 * the stream has reached this point). No host or device-wide synchronisation,
 * so a serving loop can append it to every captured round. The words are not
 * cleared; glance_clear_status clears them. Null status_out:
 * GLANCE_ERR_INVALID_ARG. Make the first call on a device outside any stream
 * capture: resolving the words may load the library's device code.
 */
glance_status glance_get_status(int32_t* status_out, void* stream);

/* Stream-ordered clear of every device status word (a memset each, enqueued
 * on `stream`). The words' addresses are looked up on each call with the
 * current device; the lookup enqueues nothing. As for glance_get_status, make
 * the first call on a device outside any stream capture. */
glance_status glance_clear_status(void* stream);

/* ABI version: major * 10000 + minor * 100 + patch. */
int glance_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GLANCE_H */
