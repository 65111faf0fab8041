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
  size_t node, tok, cls, rptr, cptr, ridx, cidx, rord, cord, hmin, hmax, runs, nruns, cnt, total;
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

// a2: one thread per packed token (padding included).  The token's node is the last node
// in preorder whose first token is <= t (zero-length nodes share their successor's start).
__global__ void k_plan_expand(PlanDev P) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int Np = P.T * TILE;
  if (t >= Np) return;
  if (t >= P.N) {
    P.tok_node[t] = -1; P.pos[t] = 0; P.g[t] = 0; P.w[t] = 0.f;
    P.tok_in[t] = -1; P.tok_out[t] = -2; P.hi[t] = -1;
    return;
  }
  int lo = 0, hi = P.n - 1;                 // largest k with dfs_tok_start[k] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.dfs_tok_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int v = P.order[lo];
  const int gv = P.leaves[v];
  P.tok_node[t] = v;
  P.pos[t] = P.pos0 + P.depth_off[v] + (t - P.tok_start[v]);
  P.g[t] = gv;
  P.w[t] = __fdiv_rn(static_cast<float>(gv), static_cast<float>(P.K));
  P.tok_in[t] = P.dfs_in[v];
  P.tok_out[t] = P.dfs_out[v];
  P.hi[t] = P.sub_end[v] - 1;
}

// per key tile: min and max of hi over its real tokens
__global__ void k_tile_hi_range(const int32_t* hi, int N, int32_t* hmin, int32_t* hmax) {
  const int kt = blockIdx.x;
  const int j = kt * TILE + threadIdx.x;
  int mn = 0x7fffffff, mx = -1;
  if (j < N) { mn = hi[j]; mx = hi[j]; }
  for (int o = 16; o; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __shared__ int smn[TILE / 32], smx[TILE / 32];
  if ((threadIdx.x & 31) == 0) { smn[threadIdx.x >> 5] = mn; smx[threadIdx.x >> 5] = mx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < TILE / 32; ++i) { mn = min(mn, smn[i]); mx = max(mx, smx[i]); }
    hmin[kt] = mn;
    hmax[kt] = mx;
  }
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

// a3: one block per query tile: classes of its row, row count, global tallies
__global__ void k_tile_rows(int N, int T, const int32_t* hmin, const int32_t* hmax, uint8_t* cls,
                            int32_t* row_cnt /* row_ptr + 1 */, int32_t* counts) {
  const int qt = blockIdx.x;
  int nnz = 0, nfull = 0;
  for (int kt = threadIdx.x; kt < T; kt += blockDim.x) {
    const uint8_t c = tile_class_of(qt, kt, N, hmin, hmax);
    cls[(size_t)qt * T + kt] = c;
    nnz += (c != 0);
    nfull += (c == 2);
  }
  for (int o = 16; o; o >>= 1) {
    nnz += __shfl_xor_sync(0xffffffffu, nnz, o);
    nfull += __shfl_xor_sync(0xffffffffu, nfull, o);
  }
  __shared__ int s_nnz[32], s_full[32];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { s_nnz[w] = nnz; s_full[w] = nfull; }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0, b = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) { a += s_nnz[i]; b += s_full[i]; }
    row_cnt[qt] = a;
    atomicAdd(&counts[0], a);
    atomicAdd(&counts[1], b);
    atomicAdd(&counts[2], a - b);
  }
}

__global__ void k_tile_cols(int N, int T, const int32_t* hmin, const int32_t* hmax,
                            int32_t* col_cnt /* col_ptr + 1 */) {
  const int kt = blockIdx.x;
  int nnz = 0;
  for (int qt = kt + threadIdx.x; qt < T; qt += blockDim.x) nnz += (tile_class_of(qt, kt, N, hmin, hmax) != 0);
  for (int o = 16; o; o >>= 1) nnz += __shfl_xor_sync(0xffffffffu, nnz, o);
  __shared__ int s[32];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = nnz;
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) a += s[i];
    col_cnt[kt] = a;
  }
}

// single block: counts -> exclusive prefix sums (in place), and heaviest-first orders
__global__ void k_tile_scan_order(int T, int32_t* row_ptr, int32_t* col_ptr, int32_t* row_order,
                                  int32_t* col_order, const int32_t* hmax) {
  __shared__ int carry[2];
  __shared__ int warp_sum[2][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  // ranks first (needs the raw counts, held in ptr[1..T])
  // rows: descending count; columns: descending last query tile (hi_max / 128), then
  // descending count; ties by ascending index
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const int rc = row_ptr[i + 1], cc = col_ptr[i + 1], cl = hmax[i] / TILE;
    int rr = 0, cr = 0;
    for (int j = 0; j < T; ++j) {
      const int rj = row_ptr[j + 1], cj = col_ptr[j + 1], lj = hmax[j] / TILE;
      rr += (rj > rc) || (rj == rc && j < i);
      cr += (lj > cl) || (lj == cl && (cj > cc || (cj == cc && j < i)));
    }
    row_order[rr] = i;
    col_order[cr] = i;
  }
  __syncthreads();
  if (threadIdx.x == 0) { carry[0] = 0; carry[1] = 0; row_ptr[0] = 0; col_ptr[0] = 0; }
  __syncthreads();
  for (int base = 0; base < T; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int a = (i < T) ? row_ptr[i + 1] : 0;
    int b = (i < T) ? col_ptr[i + 1] : 0;
    for (int o = 1; o < 32; o <<= 1) {                    // inclusive warp scan
      const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) { a += ya; b += yb; }
    }
    if (lane == 31) { warp_sum[0][w] = a; warp_sum[1][w] = b; }
    __syncthreads();
    int pa = carry[0], pb = carry[1];
    for (int k = 0; k < w; ++k) { pa += warp_sum[0][k]; pb += warp_sum[1][k]; }
    __syncthreads();
    if (i < T) { row_ptr[i + 1] = a + pa; col_ptr[i + 1] = b + pb; }
    if (threadIdx.x == blockDim.x - 1) {
      int ta_ = carry[0], tb = carry[1];
      for (int k = 0; k < nw; ++k) { ta_ += warp_sum[0][k]; tb += warp_sum[1][k]; }
      carry[0] = ta_;
      carry[1] = tb;
    }
    __syncthreads();
  }
}

// one block per query tile (rows) or key tile (cols): ordered compaction of non-empty tiles
__global__ void k_tile_fill(int T, const uint8_t* cls, const int32_t* row_ptr, int32_t* row_idx,
                            const int32_t* col_ptr, int32_t* col_idx) {
  const bool cols = blockIdx.y == 1;
  const int a = blockIdx.x;
  int32_t* out = cols ? col_idx + col_ptr[a] : row_idx + row_ptr[a];
  __shared__ int warp_cnt[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int base = 0; base < T; base += blockDim.x) {
    const int b = base + threadIdx.x;
    bool nz = false;
    if (b < T) nz = cols ? cls[(size_t)b * T + a] != 0 : cls[(size_t)a * T + b] != 0;
    const unsigned m = __ballot_sync(0xffffffffu, nz);
    if (lane == 0) warp_cnt[w] = __popc(m);
    __syncthreads();
    int off = carry;
    for (int k = 0; k < w; ++k) off += warp_cnt[k];
    if (nz) out[off + __popc(m & ((1u << lane) - 1))] = b;
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = carry;
      for (int k = 0; k < (int)(blockDim.x >> 5); ++k) s += warp_cnt[k];
      carry = s;
    }
    __syncthreads();
  }
}

// One warp per tile: split the tile's 128 tokens into maximal runs of one node (a run starts
// where dfs_in changes; padding, dfs_in = -1, is one more run) and record the first
// TREE_MAX_RUNS of them with their node interval.  The kernels test the ancestor interval once
// per run instead of once per token.
__global__ void k_tile_runs(const int32_t* tok_in, const int32_t* tok_out, int32_t* runs, int32_t* nruns) {
  const int t = blockIdx.x, lane = threadIdx.x;
  const int32_t* in = tok_in + (size_t)t * TILE;
  const int32_t* out = tok_out + (size_t)t * TILE;
  int32_t* rt = runs + (size_t)t * TREE_MAX_RUNS * 4;
  __shared__ int starts[TILE + 1];
  int base = 0;
  for (int ch = 0; ch < TILE / 32; ++ch) {
    const int c = ch * 32 + lane;
    const bool head = (c == 0) || (in[c] != in[c - 1]);
    const unsigned m = __ballot_sync(0xffffffffu, head);
    if (head) starts[base + __popc(m & ((1u << lane) - 1))] = c;
    base += __popc(m);
  }
  __syncwarp();
  if (lane == 0) starts[base] = TILE;
  __syncwarp();
  for (int k = lane; k < base && k < TREE_MAX_RUNS; k += 32) {
    const int st = starts[k];
    rt[4 * k + 0] = st;
    rt[4 * k + 1] = starts[k + 1];
    rt[4 * k + 2] = in[st];
    rt[4 * k + 3] = out[st];
  }
  if (lane == 0) nruns[t] = base;
}

__global__ void k_zero_i32(int32_t* p, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0;
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
  const int Np = T * TILE;
  k_plan_expand<<<(Np + 255) / 256, 256, 0, s>>>(P);
  k_zero_i32<<<1, 32, 0, s>>>(p->counts, 4);
  k_tile_hi_range<<<T, TILE, 0, s>>>(p->hi, N, p->tile_hi_min, p->tile_hi_max);
  k_tile_runs<<<T, 32, 0, s>>>(p->tok_in, p->tok_out, p->tile_runs, p->tile_nruns);
  k_tile_rows<<<T, 256, 0, s>>>(N, T, p->tile_hi_min, p->tile_hi_max, p->tile_class, p->row_ptr + 1, p->counts);
  k_tile_cols<<<T, 256, 0, s>>>(N, T, p->tile_hi_min, p->tile_hi_max, p->col_ptr + 1);
  k_tile_scan_order<<<1, 1024, 0, s>>>(T, p->row_ptr, p->col_ptr, p->row_order, p->col_order, p->tile_hi_max);
  k_tile_fill<<<dim3(T, 2), 256, 0, s>>>(T, p->tile_class, p->row_ptr, p->row_idx, p->col_ptr, p->col_idx);
  return record_cuda(cudaGetLastError());
}

}  // extern "C"
