/*
 * tree_attn.h - C ABI of the GB300 (sm_103a) tree-masked attention library.
 *
 * What it computes (all citations are to "Tree Training 技术详解", tingdeliu.github.io):
 *   A prefix tree of token segments (section 3.1) is packed depth-first, each node's tokens
 *   once (section 3.2, X_DFS).  Token i may attend to token j iff j <= i and node(j) is
 *   node(i) or an ancestor of it (section 4.2, mask M_ij), tested here in interval form
 *   dfs_in(node j) <= dfs_in(node i) <= dfs_out(node j) (section 4.3: node DFS intervals).
 *   RoPE positions follow tree depth (section 5); g_t counts the root-to-leaf paths through
 *   token t and g_t/K is its loss weight (section 6.2).
 *
 * Conventions shared by every entry point
 *   - Every function returns int status: TREE_OK (0) or a negative TREE_ERR_* code.  No C++
 *     exception crosses this boundary.  tree_strerror() names a code; after TREE_ERR_CUDA,
 *     tree_last_cuda_error() gives the CUDA runtime's message for the calling thread.
 *   - Device pointers are caller-owned (for example allocated by PyTorch).  The library
 *     never allocates or frees device memory and never synchronizes a stream.  The one host
 *     to device copy it makes is inside tree_plan(), ordered on the given stream.
 *   - Launches are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Errors found on the device (a bounded wait that expired) are written to the int32
 *     `status_dev` word that the caller passes and reads back after synchronizing; the
 *     kernels only ever store a nonzero code there, so the caller zeroes it beforehand.
 *   - Tensors are bf16 (raw 16-bit words, tree_bf16), row-major, token-major: Q, O, dO, dQ
 *     are [N][Hq][d]; K, V, dK, dV are [N][Hkv][d], tokens in packed depth-first order
 *     (node order[0]'s tokens first; node v's tokens start at tok_start[v]).  Pointers to
 *     them must be 16-byte aligned.  Head dimension d is 64 or 128; Hq % Hkv == 0 and
 *     q head h reads kv head h / (Hq / Hkv).
 *   - N_pad = n_tiles * 128.  Per-token plan arrays and the LSE rows are N_pad long; the
 *     entries past N are padding that the library writes itself.
 *   - Only compute capability 10.3 (GB300) is accepted: TREE_ERR_ARCH otherwise.
 */
#ifndef TREE_ATTN_H
#define TREE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t tree_bf16;             /* bfloat16 bit pattern */
typedef struct CUstream_st* tree_stream_t; /* identical to cudaStream_t */

#define TREE_TILE 128                   /* query and key tile edge */
#define TREE_MAX_RUNS 16                /* node runs per tile kept in the plan's run table */

enum {
  TREE_OK = 0,
  TREE_ERR_INVALID_TREE = -1, /* parent out of range, self parent, cycle, no root,
                                 node_len < 0, token total 0 or > 2^31-1 */
  TREE_ERR_SHAPE = -2,        /* d not 64/128, Hq % Hkv != 0, non-positive heads, plan mismatch */
  TREE_ERR_ARCH = -3,         /* current device is not compute capability 10.3 */
  TREE_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
  TREE_ERR_TIMEOUT = -5,      /* a bounded device wait expired (written to status_dev) */
  TREE_ERR_ARG = -6,          /* NULL or misaligned pointer, bad size */
  TREE_ERR_SCRATCH = -7       /* problem needs more scratch than tree_attn_bwd_noalloc holds */
};

/* ---------------------------------------------------------------------------------------
 * Plan
 * -------------------------------------------------------------------------------------*/

typedef struct {
  int32_t n_nodes;    /* nodes in the tree */
  int32_t n_tokens;   /* N = sum of node lengths */
  int32_t n_tiles;    /* T = ceil(N / 128) */
  int32_t n_paths;    /* K = root-to-leaf paths (leaves of all roots) */
  int64_t max_nnz;    /* T (T + 1) / 2: capacity of row_idx / col_idx */
  int64_t plan_bytes; /* device bytes tree_plan_bind() carves the plan arrays from (the
                         arrays below plus 12 T bytes of per-tile counts tree_plan uses
                         as scratch, placed after `counts`) */
} tree_plan_info;

/* Host-side descriptor of a plan; every pointer is device memory inside the buffer given
 * to tree_plan_bind().  Per-node arrays are indexed by node id unless noted. */
typedef struct {
  /* per node [n_nodes] */
  int32_t* order;         /* depth-first preorder of node ids (children by ascending id) */
  int32_t* dfs_in;        /* preorder index of the node */
  int32_t* dfs_out;       /* preorder index of the last node of its subtree (inclusive) */
  int32_t* tok_start;     /* first packed token of the node */
  int32_t* depth_off;     /* sum of the ancestors' lengths = position of its first token */
  int32_t* leaves;        /* root-to-leaf paths through the node (g of its tokens) */
  int32_t* dfs_tok_start; /* tok_start indexed by preorder index */
  int32_t* sub_end;       /* one past the last packed token of the node's subtree */
  /* per packed token [N_pad]; entries >= N are padding */
  int32_t* tok_node;      /* node id of the token (pad: -1) */
  int32_t* pos;           /* RoPE position = depth_off + offset in node (pad: 0) */
  int32_t* g;             /* path count g_t (pad: 0) */
  int32_t* tok_in;        /* dfs_in of the token's node (pad: -1) */
  int32_t* tok_out;       /* dfs_out of the token's node (pad: -2) */
  int32_t* hi;            /* sub_end(node) - 1: last token that can see this one (pad: -1) */
  float* w;               /* g_t / K, IEEE fp32 round-to-nearest division (pad: 0) */
  /* tile table, tiles are 128 x 128: query tile qt (rows), key tile kt (columns) */
  uint8_t* tile_class;    /* [T*T] row-major [qt][kt]: 0 empty, 1 partial, 2 full */
  int32_t* row_ptr;       /* [T+1] CSR over query tiles */
  int32_t* row_idx;       /* [max_nnz] non-empty kt of each qt, ascending */
  int32_t* col_ptr;       /* [T+1] CSR over key tiles */
  int32_t* col_idx;       /* [max_nnz] non-empty qt of each kt, ascending */
  int32_t* row_order;     /* [T] query tiles by descending row count (ties: ascending) */
  int32_t* col_order;     /* [T] key tiles by descending last query tile of their column,
                             then descending column count (ties: ascending index) */
  int32_t* tile_hi_min;   /* [T] min of hi over the key tile's real tokens */
  int32_t* tile_hi_max;   /* [T] max of hi over the key tile's real tokens */
  int32_t* tile_runs;     /* [T][TREE_MAX_RUNS][4] the tile's maximal runs of tokens of one node
                             (padding counts as one node), in order: {start, end (exclusive),
                             dfs_in, dfs_out} with start/end relative to the tile; only the
                             first min(tile_nruns, TREE_MAX_RUNS) entries are written */
  int32_t* tile_nruns;    /* [T] number of runs in the tile (may exceed TREE_MAX_RUNS) */
  int32_t* counts;        /* [4] nnz, n_full, n_partial, reserved (0) */
  int32_t n_nodes, n_tokens, n_tiles, n_paths;
} tree_plan_t;

/* Validate the tree and report its sizes.  Host only, no CUDA call.
 * parent[i] is the parent id of node i (-1 for a root); node_len[i] >= 0 its token count.
 * Returns TREE_ERR_INVALID_TREE on any of the conditions listed with that code. */
int tree_plan_query(const int32_t* parent, const int32_t* node_len, int32_t n_nodes,
                    tree_plan_info* info);

/* The plan's per-node arrays, computed on the host exactly as tree_plan computes them before
 * copying them to the device (section 3.2: depth-first preorder with children by ascending id,
 * roots by ascending id; section 4.3 intervals; section 5 depth offsets; section 6.2 leaf
 * counts).  Host only, no CUDA call.  `out` is caller-owned host memory of 8 * n_nodes int32
 * and receives, n_nodes each and in this order: order, dfs_in, dfs_out, tok_start, depth_off,
 * leaves, dfs_tok_start, sub_end (the fields of tree_plan_t with the same names).  Invalid
 * trees as tree_plan_query; out == NULL -> TREE_ERR_ARG. */
int tree_plan_nodes(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, int32_t* out);

/* Carve the plan arrays out of a caller-owned device buffer of info->plan_bytes bytes
 * (256-byte aligned) and fill `plan`'s pointers and sizes.  Host only, no CUDA call. */
int tree_plan_bind(const tree_plan_info* info, void* device_buffer, tree_plan_t* plan);

/* Build the plan on `stream` (sections 3.2, 4.3, 5, 6.2 of the explainer):
 *   host:   validation, depth-first preorder (children by ascending id), dfs_in/dfs_out,
 *           tok_start, depth_off, leaves, sub_end; one async copy of these to the device;
 *   device: three launches: per-token expansion (tok_node, pos, g, w, tok_in, tok_out,
 *           hi) with the per-key-tile hi range and node runs; tile classes with per-row and
 *           per-column counts; row/column CSR lists and heaviest-first orders.
 * `plan` must come from tree_plan_bind() for the same tree.  The host arrays may be freed
 * when the call returns. */
int tree_plan(const int32_t* parent, const int32_t* node_len, int32_t n_nodes,
              const tree_plan_t* plan, tree_stream_t stream);

/* tree_plan for one partition of a larger tree (section 8.2 of the explainer): the tree given
 * is the partition (its root is the cut node), and every position is shifted by pos_offset =
 * the number of gateway tokens above it (the cut node's depth offset in the whole tree), so
 * RoPE and the inverse rotations continue the ancestors' positions.  Everything else is the
 * partition's own (its g and w count the partition's leaves: loss weights of a partitioned
 * tree come from the whole tree's plan).  pos_offset < 0 -> TREE_ERR_ARG. */
int tree_plan_offset(const int32_t* parent, const int32_t* node_len, int32_t n_nodes,
                     int32_t pos_offset, const tree_plan_t* plan, tree_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * RoPE and loss weights
 * -------------------------------------------------------------------------------------*/

/* Rotate-half RoPE at the plan's depth positions (section 5): for c < d/2,
 * angle = pos * theta^(-2c/d) in fp32, x'_c = x_c cos - x_{c+d/2} sin,
 * x'_{c+d/2} = x_{c+d/2} cos + x_c sin.  q -> qr [N][Hq][d], k -> kr [N][Hkv][d];
 * in place (qr == q, kr == k) is allowed. */
int tree_rope_fwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                  tree_bf16* qr, tree_bf16* kr, int Hq, int Hkv, int d, float theta,
                  tree_stream_t stream);

/* dO_t = (g_t / K) * U_t (section 6.2: the per-token weight of the tree loss), u and dO
 * [N][H][d] bf16; in place allowed. */
int tree_apply_weights(const tree_plan_t* plan, const tree_bf16* u, tree_bf16* dO, int H,
                       int d, tree_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Attention (section 4.2: Softmax(Q K^T / sqrt(d) + M) V, block-sparse per section 4.3)
 * -------------------------------------------------------------------------------------*/

/* Forward.  q, k: RoPE-rotated inputs; v.  Writes o [N][Hq][d] bf16 and
 * lse [Hq][N_pad] fp32 = natural log of sum_j exp(scale q_i.k_j) over visible j
 * (padding entries 0).  scale <= 0 selects 1/sqrt(d).  Only non-empty tiles are
 * computed; the mask is evaluated on partial tiles only. */
int tree_attn_fwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                  const tree_bf16* v, int Hq, int Hkv, int d, float scale, tree_bf16* o,
                  float* lse, int32_t* status_dev, tree_stream_t stream);

/* Gateway prefix of a partition (section 8.2 of the explainer): the K/V of the tokens on the
 * path from the whole tree's root down to the cut node's parent, computed (and RoPE-rotated)
 * by the partitions above and read here without recomputation.  Every token of the
 * partition sees every gateway key: they are all its ancestors.  Gateway row r is the token
 * at position r on that path. */
typedef struct {
  const tree_bf16* k;   /* [len][Hkv][d] rotated keys, path order (root first), 16-byte aligned */
  const tree_bf16* v;   /* [len][Hkv][d]                                                      */
  int32_t len;          /* gateway tokens, >= 1 (the partition's pos_offset)                 */
} tree_gateway_t;

/* tree_attn_fwd for a partition below a gateway: each query's softmax runs over the gateway
 * keys (all visible, none masked but the rows past len of the last 128-key block) and its
 * own visible keys.  `plan` is the partition's (tree_plan_offset with pos_offset = len).
 * gw == NULL or gw->len <= 0 or a null gateway pointer -> TREE_ERR_ARG. */
int tree_attn_fwd_gateway(const tree_plan_t* plan, const tree_gateway_t* gw, const tree_bf16* q,
                          const tree_bf16* k, const tree_bf16* v, int Hq, int Hkv, int d,
                          float scale, tree_bf16* o, float* lse, int32_t* status_dev,
                          tree_stream_t stream);

/* Bytes of device workspace tree_attn_bwd needs: two fp32 [Hq][N_pad] row arrays
 * (-delta * scale with delta_i = sum_c dO_ic O_ic, and -lse * log2(e)) followed by the fp32
 * dQ accumulator (Hq * d * N_pad floats, one block per head and query tile). */
size_t tree_attn_bwd_workspace(const tree_plan_t* plan, int Hq, int d);

/* Backward of tree_attn_fwd (section 6.2: gradients of shared ancestors add up).
 * Inputs as in the forward plus o, lse and dO = dL/dO [N][Hq][d].  Outputs dq [N][Hq][d],
 * dk, dv [N][Hkv][d] bf16.  With rope_theta > 0 the inverse RoPE rotation at the plan's
 * positions is applied to dq and dk, so they are gradients w.r.t. the un-rotated q, k;
 * rope_theta <= 0 returns gradients w.r.t. the rotated inputs.  dK and dV are reduced
 * on chip per key tile and written once.  `workspace` holds tree_attn_bwd_workspace()
 * bytes, 256-byte aligned; its contents need not be initialised. */
int tree_attn_bwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                  const tree_bf16* v, const tree_bf16* o, const float* lse,
                  const tree_bf16* dO, int Hq, int Hkv, int d, float scale, float rope_theta,
                  void* workspace, tree_bf16* dq, tree_bf16* dk, tree_bf16* dv,
                  int32_t* status_dev, tree_stream_t stream);

/* tree_attn_bwd for the path-averaged tree loss of "Tree Training 技术详解" section 6.2 / 12,
 * where dL/dO_t = (g_t / K) U_t: `u` [N][Hq][d] bf16 is the unweighted per-token gradient U and
 * the plan's weights w_t = g_t / K are applied inside the backward, without forming dO.  The
 * preprocess takes delta_t = sum_c U_tc O_tc and adds log2(w_t) to the -LSE log2(e) term, so the
 * probabilities the kernel forms are P w; then dS = (P w)(dP(U) - delta) and
 * dV = sum (P w)^T U equal the gradients for dO = w U up to rounding (dO = w U is never rounded
 * to bf16 here, as tree_apply_weights does).  Same arguments, workspace and errors as
 * tree_attn_bwd (plan without weights -> TREE_ERR_ARG); equivalent to tree_apply_weights
 * followed by tree_attn_bwd, with one pass over U, O fewer. */
int tree_attn_bwd_weighted(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                           const tree_bf16* v, const tree_bf16* o, const float* lse,
                           const tree_bf16* u, int Hq, int Hkv, int d, float scale,
                           float rope_theta, void* workspace, tree_bf16* dq, tree_bf16* dk,
                           tree_bf16* dv, int32_t* status_dev, tree_stream_t stream);

/* Backward of tree_attn_fwd_gateway.  Outputs as tree_attn_bwd for the partition's own tokens
 * (dq then includes the gateway keys' contribution), plus the gateway keys' gradients from
 * this partition's queries: dk_gw, dv_gw fp32 [len][Hkv][d], ADDED to what they hold (the
 * fp32 accumulator that sums the children of one cut node before the relay to the parent;
 * zero them before the first child).  dk_gw is w.r.t. the un-rotated key when
 * rope_theta > 0 (rotated back at position r for row r).  Same workspace size as
 * tree_attn_bwd for `plan`; dk_gw, dv_gw 16-byte aligned, else TREE_ERR_ARG. */
int tree_attn_bwd_gateway(const tree_plan_t* plan, const tree_gateway_t* gw, const tree_bf16* q,
                          const tree_bf16* k, const tree_bf16* v, const tree_bf16* o,
                          const float* lse, const tree_bf16* dO, int Hq, int Hkv, int d,
                          float scale, float rope_theta, void* workspace, tree_bf16* dq,
                          tree_bf16* dk, tree_bf16* dv, float* dk_gw, float* dv_gw,
                          int32_t* status_dev, tree_stream_t stream);

/* The relay of section 8.2: add the fp32 gateway gradients accumulated over a cut node's
 * children into the parent partition's bf16 dk, dv [N_parent][Hkv][d]:
 * dk[rows[r]] += dk_gw[r] (and dv) for r < len, computed in fp32 and rounded once.
 * rows: device int32 [len], the parent-partition token index of gateway row r (distinct).
 * Pointers 16-byte aligned, else TREE_ERR_ARG. */
int tree_relay_add(const int32_t* rows, int32_t len, const float* dk_gw, const float* dv_gw,
                   int Hkv, int d, tree_bf16* dk, tree_bf16* dv, tree_stream_t stream);

/* dst[r] = src[rows[r]] for r < n: bf16 rows of row_elems elements (a multiple of 8), e.g.
 * the gateway K/V of a child partition gathered from the parent partition's rotated k and v
 * (row_elems = Hkv * d).  rows: device int32 [n]; src, dst 16-byte aligned, else
 * TREE_ERR_ARG. */
int tree_gather_rows(const int32_t* rows, int32_t n, const tree_bf16* src, tree_bf16* dst,
                     int row_elems, tree_stream_t stream);

/* Backward without any allocation by the caller or the library (this entry point has no
 * counterpart in the Tree Training explainer; it exists for callers).  Some callers cannot
 * provide the workspace tree_attn_bwd needs: code that drives this library through the plain
 * C ABI from a host runtime which owns every device allocation and forbids new ones after
 * start-up (fixed memory budgets), or that must not pay cudaMalloc's implicit device
 * synchronisation on its path.  This variant takes the delta / fp32 dQ scratch from one
 * fixed array of TREE_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library as device
 * memory; every GPU that loads the library holds that array until the process exits.
 * Same arguments and results as tree_attn_bwd, minus `workspace`.
 *   - Size limit: a problem whose tree_attn_bwd_workspace() exceeds the array is rejected
 *     with TREE_ERR_SCRATCH before anything is launched (at d = 128, Hq = 32 that is about
 *     4000 tokens).
 *   - Set-up: every call looks up the array's device address in the current device's
 *     context (a host-side symbol lookup, no allocation), so the address stays right after
 *     cudaDeviceReset.  The first call on a device may load the library's device code into
 *     that context: make it before any stream capture.
 *   - Sharing: every call on a device uses the same array, which keeps the last call's
 *     contents (the accumulator is cleared at the start of each call).  Calls that overlap
 *     on the GPU (different streams, or different host threads without ordering) race on
 *     it and corrupt each other's gradients: serialise them.
 *   - It calls no cudaMalloc / cudaFree and no allocating library routine. */
#define TREE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int tree_attn_bwd_noalloc(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                          const tree_bf16* v, const tree_bf16* o, const float* lse,
                          const tree_bf16* dO, int Hq, int Hkv, int d, float scale,
                          float rope_theta, tree_bf16* dq, tree_bf16* dk, tree_bf16* dv,
                          int32_t* status_dev, tree_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Hybrid layers over the packed tree ("Tree Training 技术详解", section 9).  In depth-first packing the
 * token before a node's first token belongs to the previous node in preorder, not to the
 * node's parent; layers that carry context along the sequence must take it from the parent.
 * parent, node_len: the tree as given to tree_plan, as device int32 arrays [n_nodes].
 * -------------------------------------------------------------------------------------*/

/* Causal depthwise convolution along root paths (section 9.2):
 *   y[t][c] = bias[c] + sum_{k < K} w[k][c] * x[prev_k(t)][c],
 * prev_0(t) = t and prev_k(t) the token k steps before t on its root path: earlier tokens of
 * t's node, then the last tokens of its parent (the nearest ancestor holding tokens), and so
 * on; terms before the root are zero.  Every token gets what a causal convolution over any
 * root-to-leaf path through it gives.  x, y [N][C] bf16 in packed order; w [K][C] fp32; bias
 * [C] fp32 or NULL.  C a multiple of 8, 1 <= K <= 8 (else TREE_ERR_SHAPE); pointers 16-byte
 * aligned (else TREE_ERR_ARG).  status_dev (device int32, may be NULL) receives
 * TREE_ERR_TIMEOUT if a wait for a staged tile runs past the wait limit, as for tree_attn_fwd. */
int tree_conv1d_fwd(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len,
                    const tree_bf16* x, const float* w, const float* bias, int C, int K,
                    tree_bf16* y, int32_t* status_dev, tree_stream_t stream);

/* Bytes of workspace tree_conv1d_bwd needs: an fp32 [N][C] array of which it uses only the
 * last K-1 rows of each node (the rows that also receive terms from the node's descendants). */
size_t tree_conv1d_bwd_workspace(const tree_plan_t* plan, int C);

/* Backward of tree_conv1d_fwd for an upstream gradient dy [N][C] bf16: dx [N][C] bf16 (each
 * x[j] collects w[k] dy[t] from every t with prev_k(t) = j: a node's last tokens feed all its
 * children), dw [K][C] and, if dbias is not NULL, dbias [C] fp32 (overwritten).  A dx row
 * inside a node gathers its K terms in a fixed order (deterministic); the last K-1 rows of a
 * node, dw and dbias are fp32 atomic sums, whose rounding order (not value) varies between runs.
 * Same shape and pointer rules as tree_conv1d_fwd; the workspace 16-byte aligned. */
int tree_conv1d_bwd(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len,
                    const tree_bf16* x, const float* w, const tree_bf16* dy, int C, int K,
                    void* workspace, tree_bf16* dx, float* dw, float* dbias, int32_t* status_dev,
                    tree_stream_t stream);

/* Recurrent-state routing (section 9.1): init[v] = final[a(v)], a(v) the nearest ancestor of
 * node v that holds tokens (zeros for roots), fp32 [n_nodes][S], S a multiple of 4. */
int tree_route_states(const int32_t* parent, const int32_t* node_len, int32_t n_nodes,
                      const float* final_states, int S, float* init_states, tree_stream_t stream);

/* Its backward: d_final[a(v)] += d_init[v] for every node v with such an ancestor (a parent
 * receives the sum over its children); d_final is accumulated into, not overwritten. */
int tree_route_states_bwd(const int32_t* parent, const int32_t* node_len, int32_t n_nodes,
                          const float* d_init, int S, float* d_final, tree_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Loss: the tree's next-token cross-entropy fused with the vocabulary projection
 * ("Tree Training 技术详解", sections 6.2, 6.3 and 12).  Each root-to-leaf path is a sequence
 * whose tokens' logits predict the next token's label; the tree loss is the average of the
 * paths' summed losses.  Equivalently, token u (label not ignore_index) is predicted by the
 * logits row z_t = W h_t of t = prev(u), the token before u on its root path (u-1 inside a
 * node; the parent's last token - nearest ancestor holding tokens - for a node's first token),
 * with weight g_u / K (the plan's w); a root's first token is predicted by nothing.
 * -------------------------------------------------------------------------------------*/

/* Workspace bytes for tree_ce_fwd_bwd: per-token pairs, label logits, weight sums and LSE,
 * plus one chunk's (max, sum exp) partials and bf16 logits gradients (chunk x V x 2 bytes). */
size_t tree_ce_workspace(const tree_plan_t* plan, int D, int V, int chunk);

/* Loss and gradients in one call, processed in chunks of `chunk` logits rows (a multiple of
 * 128; the last chunk may be shorter).  Per chunk the logits GEMM runs twice (for the row
 * logsumexp, then for the gradient), so no logits are stored; then dh rows = dz W and
 * dW (+)= dz^T h.  Inputs: h [N][D] bf16 hidden states in packed order, W [V][D] bf16,
 * labels [N] int32 (ignore_index or 0 <= y < V; any other value sets TREE_ERR_ARG in
 * status_dev and is ignored).  Outputs: *loss (device fp32 scalar), lse [N] fp32 per-row
 * logsumexp (may be NULL), dh [N][D] bf16, dW [V][D] fp32 (overwritten).  D a multiple of
 * 256, V a multiple of 8 (else TREE_ERR_SHAPE); pointers 16-byte aligned (else
 * TREE_ERR_ARG).  Rounding: logits and all sums in fp32, the logits gradient stored in bf16,
 * the loss summed in fp64. */
int tree_ce_fwd_bwd(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len,
                    const tree_bf16* h, const tree_bf16* W, const int32_t* labels, int D, int V,
                    int chunk, int ignore_index, void* workspace, float* loss, float* lse,
                    tree_bf16* dh, float* dW, int32_t* status_dev, tree_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Diagnostics
 * -------------------------------------------------------------------------------------*/

/* The GEMM kernel behind tree_ce_fwd_bwd on its own: C [M][N] fp32 = op(A) op(B)^T with
 * a_mn = 0: A stored [M][K], 1: A stored [K][M]; b_mn = 0: B stored [N][K], 1: B stored
 * [K][N] (bf16, row-major).  M, N, K multiples of 8; pointers 16-byte aligned. */
int tree_diag_gemm(const tree_bf16* A, const tree_bf16* B, int M, int N, int K, int a_mn, int b_mn,
                   float* C, int32_t* status_dev, tree_stream_t stream);

/* CTAs per key-tile column in the backward (1, 2 or 4; 0 = automatic, the default).  A split
 * column runs as a thread-block cluster: CTA r of the cluster takes the column's steps
 * r, r + s, r + 2s, ... (s = the split) and the cluster sums its fp32 dK / dV partials through
 * distributed shared memory, in rank order, before the single write-out (deterministic).
 * Automatic: the largest of 1, 2, 4 for which the split grid (key tiles x kv heads x split)
 * still fits one wave of SMs, i.e. only trees too small to occupy the GPU are split (a cluster
 * needs all its SMs free at once, which costs throughput on a busy GPU: measured no gain for
 * 216 columns on 152 SMs).  Process-wide; for tests and measurements.  Other values ->
 * TREE_ERR_ARG. */
int tree_set_bwd_split(int split);

/* CTAs per query-tile row in the forward (1, 2 or 4; 0 = automatic, the default): split-KV.  A
 * split row runs as a thread-block cluster: CTA r of the cluster takes the row's key tiles
 * r, r + s, r + 2s, ... (gateway tiles included) with its own online-softmax state (m, l, O),
 * and rank 0 merges the states by the Tree Attention page's associative rule
 * (m = max m_r, l = sum l_r 2^(m_r - m), O = sum O_r 2^(m_r - m)) read through distributed
 * shared memory before writing O / l and the LSE.  Automatic: the largest of 1, 2, 4 for which
 * the grid (query tiles x q-head pairs x split) fits one wave of SMs (e.g. a small partition
 * below a long gateway: 256 tokens below 32768, forward 444 -> 174 us).  Process-wide.  Other
 * values -> TREE_ERR_ARG. */
int tree_set_fwd_split(int split);

/* Device waits give up after this many nanoseconds and report TREE_ERR_TIMEOUT
 * (default 2e9).  Values < 1e5 are raised to 1e5.  Process-wide. */
int tree_set_wait_limit_ns(int64_t ns);

/* Launch one kernel that waits on a barrier nobody arrives at, with a limit of `ns`
 * nanoseconds; it must store TREE_ERR_TIMEOUT into *status_dev and exit normally.
 * Exercises the bounded-wait path without faulting or hanging the GPU. */
int tree_selftest_timeout(int32_t* status_dev, int64_t ns, tree_stream_t stream);

/* Register up to 4 cudaEvent_t handles (created by the caller on the current device) that
 * tree_attn_bwd records on its stream: [0] before the delta/zeroing kernels, [1] before the
 * dK/dV kernel, [2] after it, [3] after the dQ finalize kernel.  n = 0 unregisters.  For
 * per-kernel timing with CUDA events; process-wide, not thread-safe. */
int tree_set_timing_events(void* const* events, int n);

const char* tree_strerror(int code);
const char* tree_last_cuda_error(void);
int tree_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TREE_ATTN_H */
