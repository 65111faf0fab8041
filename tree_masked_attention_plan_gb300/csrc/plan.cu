// tree_plan: the node pass on the host, then per-token expansion and the 128x128 tile table
// on the device ("Tree Training 技术详解": section 3.2 DFS serialization, section 4.3 node DFS
// intervals and ancestor block table, section 5 depth positions, section 6.2 path counts).
#include <cstdlib>
#include <cstring>
#include <vector>

#include "common.cuh"

namespace ta {
namespace {

constexpr int64_t kInt32Max = 2147483647LL;

struct NodePass {
  int n = 0, N = 0, T = 0, K = 0;
  // per node, 8 arrays in the device order of the node block
  std::vector<int32_t> block;   // [8 * n]: order, dfs_in, dfs_out, tok_start, depth_off, leaves,
                                //          dfs_tok_start, sub_end
};

// Validation and depth-first preorder with children in ascending id, roots in ascending id.
int node_pass(const int32_t* parent, const int32_t* node_len, int32_t n, NodePass* out) {
  if (!parent || !node_len || n <= 0) return n <= 0 ? TREE_ERR_INVALID_TREE : TREE_ERR_ARG;
  std::vector<int32_t> child_cnt(n + 1, 0), child_ptr(n + 1, 0), child(n);
  int64_t total = 0;
  int roots = 0;
  for (int i = 0; i < n; ++i) {
    const int32_t p = parent[i];
    if (p < -1 || p >= n || p == i) return TREE_ERR_INVALID_TREE;
    if (node_len[i] < 0) return TREE_ERR_INVALID_TREE;
    total += node_len[i];
    if (p == -1) ++roots; else ++child_cnt[p];
  }
  if (roots == 0 || total <= 0 || total > kInt32Max) return TREE_ERR_INVALID_TREE;
  for (int i = 0; i < n; ++i) child_ptr[i + 1] = child_ptr[i] + child_cnt[i];
  {
    std::vector<int32_t> fill(child_ptr.begin(), child_ptr.end() - 1);
    for (int c = 0; c < n; ++c)                 // ascending c keeps each child list ascending
      if (parent[c] >= 0) child[fill[parent[c]]++] = c;
  }
  out->n = n;
  out->block.assign(8 * (size_t)n, 0);
  int32_t* order = out->block.data();
  int32_t* dfs_in = order + n;
  int32_t* dfs_out = order + 2 * n;
  int32_t* tok_start = order + 3 * n;
  int32_t* depth_off = order + 4 * n;
  int32_t* leaves = order + 5 * n;
  int32_t* dfs_tok_start = order + 6 * n;
  int32_t* sub_end = order + 7 * n;
  std::vector<int32_t> next_child(n, 0);
  std::vector<int32_t> stack;
  stack.reserve(64);
  int pre = 0;
  int64_t tok = 0;
  for (int r = 0; r < n; ++r) {
    if (parent[r] != -1) continue;
    // enter r
    stack.push_back(r);
    dfs_in[r] = pre; order[pre] = r; dfs_tok_start[pre] = (int32_t)tok; ++pre;
    tok_start[r] = (int32_t)tok; depth_off[r] = 0; tok += node_len[r];
    while (!stack.empty()) {
      const int v = stack.back();
      const int k = next_child[v];
      if (k < child_cnt[v]) {
        next_child[v] = k + 1;
        const int c = child[child_ptr[v] + k];
        stack.push_back(c);
        dfs_in[c] = pre; order[pre] = c; dfs_tok_start[pre] = (int32_t)tok; ++pre;
        tok_start[c] = (int32_t)tok;
        depth_off[c] = depth_off[v] + node_len[v];
        tok += node_len[c];
      } else {                                          // leave v
        stack.pop_back();
        dfs_out[v] = pre - 1;
        sub_end[v] = (int32_t)tok;
        int32_t lv = 0;
        for (int j = child_ptr[v]; j < child_ptr[v + 1]; ++j) lv += leaves[child[j]];
        leaves[v] = child_cnt[v] == 0 ? 1 : lv;
      }
    }
  }
  if (pre != n) return TREE_ERR_INVALID_TREE;            // nodes on a cycle are never reached
  int64_t K = 0;
  for (int r = 0; r < n; ++r)
    if (parent[r] == -1) K += leaves[r];
  if (K > kInt32Max) return TREE_ERR_INVALID_TREE;
  out->N = (int)total;
  out->T = (int)((total + TILE - 1) / TILE);
  out->K = (int)K;
  return TREE_OK;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t node, tok, cls, rptr, cptr, ridx, cidx, rord, cord, hmin, hmax, runs, nruns, cnt, tcnt, total;
};

Layout layout(int n, int N, int T) {
  const size_t Np = (size_t)T * TILE;
  const size_t nnz = (size_t)T * (T + 1) / 2;
  Layout L{};
  size_t o = 0;
  L.node = o; o += align256(8 * (size_t)n * 4);
  L.tok = o;  o += 7 * align256(Np * 4);
  L.cls = o;  o += align256((size_t)T * T);
  L.rptr = o; o += align256((T + 1) * 4);
  L.cptr = o; o += align256((T + 1) * 4);
  L.ridx = o; o += align256(nnz * 4);
  L.cidx = o; o += align256(nnz * 4);
  L.rord = o; o += align256(T * 4);
  L.cord = o; o += align256(T * 4);
  L.hmin = o; o += align256(T * 4);
  L.hmax = o; o += align256(T * 4);
  L.runs = o; o += align256((size_t)T * TREE_MAX_RUNS * 16);
  L.nruns = o; o += align256(T * 4);
  L.cnt = o;  o += align256(4 * 4);
  L.tcnt = o; o += align256(3 * (size_t)T * 4);   // row count, row full, column count
  L.total = o;
  (void)N;
  return L;
}

// ------------------------------------------------------------------------------------------
// device kernels

struct PlanDev {
  const int32_t *order, *dfs_in, *dfs_out, *tok_start, *depth_off, *leaves, *dfs_tok_start, *sub_end;
  int32_t *tok_node, *pos, *g, *tok_in, *tok_out, *hi;
  float* w;
  int n, N, T, K;
  int pos0;                 // position of the first token of every root (0, or a gateway's length)
};

// Sum of `v` over the block (blockDim.x a multiple of 32, at most 1024 threads); every thread
// gets the result.  `red` is shared scratch of 32 ints; the call ends with a barrier so the
// scratch may be reused at once.
__device__ __forceinline__ int block_sum(int v, int* red) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  int s = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
  __syncthreads();
  return s;
}

// Launch 1 (a2 + per key tile data): one block of 128 threads per tile, one thread per packed
// token (padding included).  A token's node is the last node in preorder whose first token is
// <= t (zero-length nodes share their successor's start).  The block then reduces the tile's
// hi range over its real tokens and splits the tile into maximal runs of one node (a run starts
// where dfs_in changes; padding, dfs_in = -1, is one more run), recording the first
// TREE_MAX_RUNS runs with their node interval: the attention kernels test the ancestor interval
// once per run instead of once per token.
__global__ void __launch_bounds__(TILE) k_plan_tokens(PlanDev P, int32_t* hmin, int32_t* hmax, int32_t* runs,
                                                      int32_t* nruns) {
  const int kt = blockIdx.x, c = threadIdx.x;
  const int t = kt * TILE + c;
  __shared__ int s_in[TILE], s_out[TILE];
  __shared__ int s_mn[TILE / 32], s_mx[TILE / 32];
  __shared__ int starts[TILE + 1];
  __shared__ int s_nrun;
  int tin = -1, tout = -2, hi = -1;
  if (t >= P.N) {
    P.tok_node[t] = -1; P.pos[t] = 0; P.g[t] = 0; P.w[t] = 0.f;
    P.tok_in[t] = -1; P.tok_out[t] = -2; P.hi[t] = -1;
  } else {
    int lo = 0, up = P.n - 1;                 // largest k with dfs_tok_start[k] <= t
    while (lo < up) {
      const int mid = (lo + up + 1) >> 1;
      if (P.dfs_tok_start[mid] <= t) lo = mid; else up = mid - 1;
    }
    const int v = P.order[lo];
    const int gv = P.leaves[v];
    tin = P.dfs_in[v];
    tout = P.dfs_out[v];
    hi = P.sub_end[v] - 1;
    P.tok_node[t] = v;
    P.pos[t] = P.pos0 + P.depth_off[v] + (t - P.tok_start[v]);
    P.g[t] = gv;
    P.w[t] = __fdiv_rn(static_cast<float>(gv), static_cast<float>(P.K));
    P.tok_in[t] = tin;
    P.tok_out[t] = tout;
    P.hi[t] = hi;
  }
  s_in[c] = tin;
  s_out[c] = tout;
  // hi range over the real tokens (none: INT_MAX, -1)
  int mn = t < P.N ? hi : 0x7fffffff, mx = t < P.N ? hi : -1;
  for (int o = 16; o; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if ((c & 31) == 0) { s_mn[c >> 5] = mn; s_mx[c >> 5] = mx; }
  __syncthreads();
  if (c < 32) {                               // warp 0: range, then the run starts in order
    const int lane = c;
    if (lane == 0) {
      for (int i = 1; i < TILE / 32; ++i) { mn = min(mn, s_mn[i]); mx = max(mx, s_mx[i]); }
      hmin[kt] = min(mn, s_mn[0]);
      hmax[kt] = max(mx, s_mx[0]);
    }
    int base = 0;
    for (int ch = 0; ch < TILE / 32; ++ch) {
      const int cc = ch * 32 + lane;
      const bool head = (cc == 0) || (s_in[cc] != s_in[cc - 1]);
      const unsigned m = __ballot_sync(0xffffffffu, head);
      if (head) starts[base + __popc(m & ((1u << lane) - 1))] = cc;
      base += __popc(m);
    }
    if (lane == 0) { starts[base] = TILE; s_nrun = base; }
  }
  __syncthreads();
  const int nr = s_nrun;
  int32_t* rt = runs + (size_t)kt * TREE_MAX_RUNS * 4;
  if (c < nr && c < TREE_MAX_RUNS) {
    const int st = starts[c];
    rt[4 * c + 0] = st;
    rt[4 * c + 1] = starts[c + 1];
    rt[4 * c + 2] = s_in[st];
    rt[4 * c + 3] = s_out[st];
  }
  if (c == 0) nruns[kt] = nr;
}

// Class of tile (qt, kt).  With hi[j] the last token of node(j)'s subtree, token i sees j
// iff j <= i <= hi[j] (the interval test of section 4.3 on a depth-first packing).
__device__ __forceinline__ uint8_t tile_class_of(int qt, int kt, int N, const int32_t* hmin,
                                                 const int32_t* hmax) {
  if (kt > qt) return 0;
  if (kt == qt) return 1;                        // the diagonal always holds i == j, never all
  const int q0 = qt * TILE;
  if (hmax[kt] < q0) return 0;                   // no key of the tile reaches the first query
  if (q0 + TILE - 1 < N && hmin[kt] >= q0 + TILE - 1) return 2;
  return 1;
}

// Launch 2 (a3 classes): block a writes row a of the class table and counts the non-empty and
// full tiles of row a and the non-empty tiles of column a.
__global__ void __launch_bounds__(256) k_plan_classes(int N, int T, const int32_t* hmin, const int32_t* hmax,
                                                      uint8_t* cls, int32_t* row_cnt, int32_t* row_full,
                                                      int32_t* col_cnt) {
  __shared__ int red[32];
  const int a = blockIdx.x;
  int rn = 0, rf = 0, cn = 0;
  for (int b = threadIdx.x; b < T; b += blockDim.x) {
    const uint8_t c = tile_class_of(a, b, N, hmin, hmax);
    cls[(size_t)a * T + b] = c;
    rn += (c != 0);
    rf += (c == 2);
    cn += (tile_class_of(b, a, N, hmin, hmax) != 0);
  }
  rn = block_sum(rn, red);
  rf = block_sum(rf, red);
  cn = block_sum(cn, red);
  if (threadIdx.x == 0) { row_cnt[a] = rn; row_full[a] = rf; col_cnt[a] = cn; }
}

// Launch 3 (a3 CSR and orders): block a computes, from the per-row / per-column counts of
// launch 2, the offsets row_ptr[a], col_ptr[a] (sums over the rows / columns before a), the
// ranks of row a and column a in the heaviest-first orders (rows: count descending, then index;
// columns: last non-empty query tile descending, then count descending, then index), and
// fills row a's and column a's lists in ascending order.  The last block writes the totals.
__global__ void __launch_bounds__(256) k_plan_lists(int N, int T, const int32_t* hmin, const int32_t* hmax,
                                                    const int32_t* row_cnt, const int32_t* row_full,
                                                    const int32_t* col_cnt, int32_t* row_ptr, int32_t* row_idx,
                                                    int32_t* col_ptr, int32_t* col_idx, int32_t* row_order,
                                                    int32_t* col_order, int32_t* counts) {
  __shared__ int red[32];
  __shared__ int wrow[32], wcol[32];
  const int a = blockIdx.x;
  const int ra = row_cnt[a], ca = col_cnt[a], la = hmax[a] / TILE;
  int pr = 0, pc = 0, rr = 0, cr = 0, tf = 0;
  for (int j = threadIdx.x; j < T; j += blockDim.x) {
    const int rj = row_cnt[j], cj = col_cnt[j], lj = hmax[j] / TILE;
    if (j < a) { pr += rj; pc += cj; }
    rr += (rj > ra) || (rj == ra && j < a);
    cr += (lj > la) || (lj == la && (cj > ca || (cj == ca && j < a)));
    tf += row_full[j];
  }
  pr = block_sum(pr, red);
  pc = block_sum(pc, red);
  rr = block_sum(rr, red);
  cr = block_sum(cr, red);
  if (threadIdx.x == 0) {
    row_ptr[a] = pr;
    col_ptr[a] = pc;
    row_order[rr] = a;
    col_order[cr] = a;
  }
  if (a == T - 1) {
    tf = block_sum(tf, red);
    if (threadIdx.x == 0) {
      row_ptr[T] = pr + ra;
      col_ptr[T] = pc + ca;
      counts[0] = pr + ra;
      counts[1] = tf;
      counts[2] = pr + ra - tf;
      counts[3] = 0;
    }
  }
  // ordered compaction of the non-empty tiles of row a (over kt) and column a (over qt)
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int orow = pr, ocol = pc;
  for (int base = 0; base < T; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const bool nr = b < T && tile_class_of(a, b, N, hmin, hmax) != 0;
    const bool nc = b < T && tile_class_of(b, a, N, hmin, hmax) != 0;
    const unsigned mr = __ballot_sync(0xffffffffu, nr), mc = __ballot_sync(0xffffffffu, nc);
    if (lane == 0) { wrow[w] = __popc(mr); wcol[w] = __popc(mc); }
    __syncthreads();
    int offr = orow, offc = ocol, totr = 0, totc = 0;
    for (int k = 0; k < nw; ++k) {
      if (k < w) { offr += wrow[k]; offc += wcol[k]; }
      totr += wrow[k];
      totc += wcol[k];
    }
    const unsigned below = (1u << lane) - 1;
    if (nr) row_idx[offr + __popc(mr & below)] = b;
    if (nc) col_idx[offc + __popc(mc & below)] = b;
    orow += totr;
    ocol += totc;
    __syncthreads();
  }
}

}  // namespace
}  // namespace ta

using namespace ta;

extern "C" {

int tree_plan_query(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, tree_plan_info* info) {
  if (!info) return TREE_ERR_ARG;
  NodePass np;
  const int rc = node_pass(parent, node_len, n_nodes, &np);
  if (rc) return rc;
  info->n_nodes = np.n;
  info->n_tokens = np.N;
  info->n_tiles = np.T;
  info->n_paths = np.K;
  info->max_nnz = (int64_t)np.T * (np.T + 1) / 2;
  info->plan_bytes = (int64_t)layout(np.n, np.N, np.T).total;
  return TREE_OK;
}

int tree_plan_nodes(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, int32_t* out) {
  if (!out) return TREE_ERR_ARG;
  NodePass np;
  const int rc = node_pass(parent, node_len, n_nodes, &np);
  if (rc) return rc;
  std::memcpy(out, np.block.data(), np.block.size() * sizeof(int32_t));
  return TREE_OK;
}

int tree_plan_bind(const tree_plan_info* info, void* buf, tree_plan_t* p) {
  if (!info || !p || !buf || (reinterpret_cast<uintptr_t>(buf) & 255) != 0) return TREE_ERR_ARG;
  const int n = info->n_nodes, N = info->n_tokens, T = info->n_tiles;
  if (n <= 0 || N <= 0 || T != (N + TILE - 1) / TILE) return TREE_ERR_SHAPE;
  const Layout L = layout(n, N, T);
  char* b = static_cast<char*>(buf);
  int32_t* node = reinterpret_cast<int32_t*>(b + L.node);
  p->order = node; p->dfs_in = node + n; p->dfs_out = node + 2 * n; p->tok_start = node + 3 * n;
  p->depth_off = node + 4 * n; p->leaves = node + 5 * n; p->dfs_tok_start = node + 6 * n;
  p->sub_end = node + 7 * n;
  const size_t tstride = align256((size_t)T * TILE * 4);
  char* tk = b + L.tok;
  p->tok_node = reinterpret_cast<int32_t*>(tk + 0 * tstride);
  p->pos = reinterpret_cast<int32_t*>(tk + 1 * tstride);
  p->g = reinterpret_cast<int32_t*>(tk + 2 * tstride);
  p->tok_in = reinterpret_cast<int32_t*>(tk + 3 * tstride);
  p->tok_out = reinterpret_cast<int32_t*>(tk + 4 * tstride);
  p->hi = reinterpret_cast<int32_t*>(tk + 5 * tstride);
  p->w = reinterpret_cast<float*>(tk + 6 * tstride);
  p->tile_class = reinterpret_cast<uint8_t*>(b + L.cls);
  p->row_ptr = reinterpret_cast<int32_t*>(b + L.rptr);
  p->col_ptr = reinterpret_cast<int32_t*>(b + L.cptr);
  p->row_idx = reinterpret_cast<int32_t*>(b + L.ridx);
  p->col_idx = reinterpret_cast<int32_t*>(b + L.cidx);
  p->row_order = reinterpret_cast<int32_t*>(b + L.rord);
  p->col_order = reinterpret_cast<int32_t*>(b + L.cord);
  p->tile_hi_min = reinterpret_cast<int32_t*>(b + L.hmin);
  p->tile_hi_max = reinterpret_cast<int32_t*>(b + L.hmax);
  p->tile_runs = reinterpret_cast<int32_t*>(b + L.runs);
  p->tile_nruns = reinterpret_cast<int32_t*>(b + L.nruns);
  p->counts = reinterpret_cast<int32_t*>(b + L.cnt);
  p->n_nodes = n; p->n_tokens = N; p->n_tiles = T; p->n_paths = info->n_paths;
  return TREE_OK;
}

int tree_plan(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, const tree_plan_t* p,
              tree_stream_t stream_) {
  return tree_plan_offset(parent, node_len, n_nodes, 0, p, stream_);
}

int tree_plan_offset(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, int32_t pos_offset,
                     const tree_plan_t* p, tree_stream_t stream_) {
  if (!p || pos_offset < 0) return TREE_ERR_ARG;
  NodePass np;
  int rc = node_pass(parent, node_len, n_nodes, &np);
  if (rc) return rc;
  if (np.n != p->n_nodes || np.N != p->n_tokens || np.T != p->n_tiles || np.K != p->n_paths)
    return TREE_ERR_SHAPE;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_);
  const int n = np.n, N = np.N, T = np.T;
  // the 8 per-node arrays are contiguous in the bound layout: one copy
  rc = record_cuda(cudaMemcpyAsync(p->order, np.block.data(), np.block.size() * 4, cudaMemcpyHostToDevice, s));
  if (rc) return rc;
  PlanDev P{p->order, p->dfs_in, p->dfs_out, p->tok_start, p->depth_off, p->leaves, p->dfs_tok_start,
            p->sub_end, p->tok_node, p->pos, p->g, p->tok_in, p->tok_out, p->hi, p->w, n, N, T, np.K, pos_offset};
  // Three launches: tokens and per-key-tile data; classes and per-row / per-column counts; CSR
  // lists and orders.  The counts go to the scratch tree_plan_bind() lays out right after the
  // `counts` words (3 T int32: row count, row full count, column count).
  const Layout L = layout(n, N, T);
  int32_t* tcnt = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(p->counts) + (L.tcnt - L.cnt));
  k_plan_tokens<<<T, TILE, 0, s>>>(P, p->tile_hi_min, p->tile_hi_max, p->tile_runs, p->tile_nruns);
  k_plan_classes<<<T, 256, 0, s>>>(N, T, p->tile_hi_min, p->tile_hi_max, p->tile_class, tcnt, tcnt + T,
                                   tcnt + 2 * T);
  k_plan_lists<<<T, 256, 0, s>>>(N, T, p->tile_hi_min, p->tile_hi_max, tcnt, tcnt + T, tcnt + 2 * T, p->row_ptr,
                                 p->row_idx, p->col_ptr, p->col_idx, p->row_order, p->col_order, p->counts);
  return record_cuda(cudaGetLastError());
}

}  // extern "C"
