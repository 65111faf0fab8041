// Hybrid (attention + SSM) layers over the packed tree ("Tree Training 技术详解", section 9):
// in depth-first packing the token before a node's first token is the last token of the
// previous node in preorder, not of the node's parent, so layers that carry state along the
// sequence must read it from the parent instead.
//   * causal convolution (section 9.2): y_t = bias + sum_k w_k * x_{prev_k(t)}, where prev_k(t)
//     is the token k steps before t on its root path (the parent's last tokens once t's own node
//     is exhausted; zero before the root) - the same result as running the convolution on every
//     root-to-leaf path separately;
//   * recurrent state routing (section 9.1): a node starts from the final state of its parent
//     (the nearest ancestor that holds tokens), and in the backward the parent receives the sum
//     of its children's initial-state gradients.
// All HBM-bound: 16-byte vector accesses, eight channels per thread.
#include <algorithm>

#include "common.cuh"

namespace ta {
int make_tmap_bf16_2d(CUtensorMap* m, const void* base, int inner, int rows, int box_inner, int box_rows);  // host.cu

namespace {

// Nearest ancestor of v that holds tokens, or -1.  The walk is bounded by the node count and
// stops at an out-of-range id, so a parent array that does not describe a tree cannot hang it.
DEVI int token_ancestor(int v, const int32_t* __restrict__ parent, const int32_t* __restrict__ node_len, int n) {
  int a = parent[v];
  for (int guard = 0; a >= 0 && a < n && node_len[a] == 0 && guard < n; ++guard) a = parent[a];
  return (a >= 0 && a < n && node_len[a] > 0) ? a : -1;
}

// the token one step before j on its root path, or -1 before the root
DEVI int path_prev1(int j, const int32_t* __restrict__ tok_node, const int32_t* __restrict__ tok_start,
                    const int32_t* __restrict__ parent, const int32_t* __restrict__ node_len, int n) {
  const int v = tok_node[j];
  if (j > tok_start[v]) return j - 1;
  const int a = token_ancestor(v, parent, node_len, n);
  return a < 0 ? -1 : tok_start[a] + node_len[a] - 1;
}

DEVI void load8(const uint4* p, float (&f)[8]) {
  const uint4 u = *p;
  f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
}

DEVI void red_add8(float* dst, const float (&f)[8]) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3])
               : "memory");
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4), "f"(f[4]), "f"(f[5]), "f"(f[6]),
               "f"(f[7])
               : "memory");
}

struct ConvArgs {
  const int32_t* tok_node;
  const int32_t* tok_start;
  const int32_t* parent;
  const int32_t* node_len;
  int N, C, K, n_nodes;
};

constexpr int kConvMaxK = 8;
constexpr int kConvWarps = 8;               // a block: 32 channel groups (lanes) x 8 token lanes (warps)
constexpr int kConvRowBytes = 512;          // largest staged row: 32 lanes x 8 bf16 channels (a multiple of 128)
constexpr int kConvFwdTile = 64;            // tokens per staged tile
constexpr int kConvBwdTile = 32;

DEVI void fma8(float (&acc)[8], const float (&w)[8], const float (&x)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = fmaf(w[e], x[e], acc[e]);
}

DEVI void load_w8(const float* p, float (&f)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

DEVI uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

DEVI void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// TMA tensor copies land on 128-byte boundaries: stages are rounded up to that, and the dynamic
// shared memory base is aligned up to 1024 bytes (the launch reserves the slack).
constexpr int kConvStageAlign = 128;
DEVI int round_stage(int bytes) { return (bytes + kConvStageAlign - 1) & ~(kConvStageAlign - 1); }
DEVI uint8_t* align_smem(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// After a wait gave up: give the block's copies still in flight a bounded time to land before
// the block's shared memory is released.
DEVI void drain_bar(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < limit_ns) {
  }
}

// Tile bookkeeping shared by both kernels.  A block owns one 256-channel slab (blockIdx.y) and
// walks token tiles blockIdx.x, blockIdx.x + gridDim.x, ...  Two stages: while tile i is
// computed, tile i+1's rows are in flight (one 2-D TMA load per staged tensor) and so are its
// node ids (4-byte cp.async copies, one commit group per tile).  A node's tokens are
// contiguous in packed order, so "t-k is in t's node" is ids[t-k] == ids[t]: no lookups of the
// node's extent on the fast path.
//   ids[m] = node of token T0 - (K-1) + m, or -1 outside [0, N)
DEVI void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
DEVI void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }   // all but the newest
DEVI void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

DEVI void stage_ids(const ConvArgs& a, int first, int count, int* ids) {
  for (int m = threadIdx.x; m < count; m += blockDim.x) {
    const int t = first + m;
    if (t >= 0 && t < a.N)
      cp_async4(ids + m, a.tok_node + t);
    else
      ids[m] = -1;
  }
}

// Forward.  Staged x rows [T0-(K-1), T0+TB) (rows before 0 read as zero and are never used).
// Warp w takes tokens T0+w, T0+w+8, ...; a token at offset >= K-1 in its node reads rows t-k
// from the stage, the first K-1 tokens of a node walk up the tree and read global memory.
template <int K>
__global__ void __launch_bounds__(256) k_conv_fwd(const __grid_constant__ CUtensorMap tmX, ConvArgs a,
                                                  const uint4* __restrict__ x, const float* __restrict__ w,
                                                  const float* __restrict__ bias, uint4* __restrict__ y, int rs,
                                                  int32_t* status, uint64_t limit_ns) {
  constexpr int TB = kConvFwdTile, R = TB + K - 1;
  const int BOX = R * rs;                        // rs: bytes of one staged row (512, or 2C when C < 256)
  const int STAGE = round_stage(BOX);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem(smem_raw);
  constexpr int NIDS = TB + K - 1;               // ids of rows [T0-(K-1), T0+TB)
  __shared__ uint64_t bars[2];
  __shared__ int ids[2][NIDS];
  __shared__ int abort_flag;
  const int CV = a.C / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cv = blockIdx.y * 32 + lane;
  const bool on = cv < CV;
  const int n_tiles = (a.N + TB - 1) / TB;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmX);
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, status, limit_ns};
  float wr[K][8], b[8];
#pragma unroll
  for (int k = 0; k < K; ++k) {
#pragma unroll
    for (int e = 0; e < 8; ++e) wr[k][e] = 0.f;
    if (on) load_w8(w + (size_t)k * a.C + 8 * cv, wr[k]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) b[e] = 0.f;
  if (on && bias) load_w8(bias + 8 * cv, b);
  int tile = blockIdx.x;
  if (threadIdx.x == 0 && tile < n_tiles) {
    mbar_expect_tx(&bars[0], BOX);
    tma_load_2d(smem, &tmX, &bars[0], blockIdx.y * 256, tile * TB - (K - 1));
  }
  if (tile < n_tiles) stage_ids(a, tile * TB - (K - 1), NIDS, ids[0]);
  cp_async_commit();
  int i = 0;
  bool aborted = false;
  for (; tile < n_tiles; ++i, tile += gridDim.x) {
    const int s = i & 1;
    const int next = tile + gridDim.x;
    if (next < n_tiles) {
      if (threadIdx.x == 0) {
        mbar_expect_tx(&bars[s ^ 1], BOX);
        tma_load_2d(smem + (s ^ 1) * STAGE, &tmX, &bars[s ^ 1], blockIdx.y * 256, next * TB - (K - 1));
      }
      stage_ids(a, next * TB - (K - 1), NIDS, ids[s ^ 1]);
    }
    cp_async_commit();
    cp_async_wait_prev();
    const bool ok = mbar_wait(&bars[s], (i >> 1) & 1, wc);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const uint8_t* xs = smem + s * STAGE + lane * 16;
    const int T0 = tile * TB;
    if (on) {
#pragma unroll 4
      for (int r = warp; r < TB; r += kConvWarps) {
        const int t = T0 + r;
        if (t >= a.N) break;
        float acc[8], xv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = b[e];
        if (ids[s][r] == ids[s][r + K - 1]) {     // t-K+1 .. t all in t's node
#pragma unroll
          for (int k = 0; k < K; ++k) {
            load8(reinterpret_cast<const uint4*>(xs + (r + K - 1 - k) * rs), xv);
            fma8(acc, wr[k], xv);
          }
        } else {
          int j = t;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            if (j < 0) break;
            load8(x + (size_t)j * CV + cv, xv);
            fma8(acc, wr[k], xv);
            j = path_prev1(j, a.tok_node, a.tok_start, a.parent, a.node_len, a.n_nodes);
          }
        }
        y[(size_t)t * CV + cv] = pack8(acc);
      }
    }
    __syncthreads();
  }
  cp_async_wait_all();
  if (aborted && threadIdx.x == 0) {
    drain_bar(&bars[i & 1], (i >> 1) & 1, limit_ns);
    if (tile + gridDim.x < n_tiles) drain_bar(&bars[(i & 1) ^ 1], ((i + 1) >> 1) & 1, limit_ns);
  }
}

// Backward, gathered by output row:
//   dx_j = sum_k w_k sum_{t : prev_k(t) = j} dy_t,   dw_k = sum_t x_{prev_k(t)} dy_t,   db = sum_t dy_t.
// Staged per tile: x rows [T0-(K-1), T0+TB) and dy rows [T0, T0+TB+K-1).  Inside a node
// prev_k(t) = t - k, so row j gathers dy_{j..j+K-1} from the stage and is written once, in
// bf16.  Only the last K-1 rows of a node also receive terms from its descendants (their first
// tokens reach back across the node boundary); those rows are summed in fp32 in the workspace
// - the row's own interior part and every cross-boundary term, red-added - and converted by
// k_conv_bwd_finish.  dw and db: per-thread sums over the block's tiles, reduced over the warps
// in shared memory, one red.add per block.
template <int K>
__global__ void __launch_bounds__(256) k_conv_bwd(const __grid_constant__ CUtensorMap tmX,
                                                  const __grid_constant__ CUtensorMap tmDY, ConvArgs a,
                                                  const uint4* __restrict__ x, const float* __restrict__ w, float* ws,
                                                  uint4* __restrict__ dx, float* dw, float* dbias, int rs,
                                                  int32_t* status, uint64_t limit_ns) {
  constexpr int TB = kConvBwdTile, R = TB + K - 1;
  const int BOX = R * rs;                        // rs: bytes of one staged row (512, or 2C when C < 256)
  const int HALF = round_stage(BOX), STAGE = 2 * HALF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem(smem_raw);
  constexpr int NIDS = TB + 2 * (K - 1);         // ids of rows [T0-(K-1), T0+TB+K-1)
  __shared__ uint64_t bars[2];
  __shared__ int ids[2][NIDS];
  __shared__ int abort_flag;
  __shared__ __align__(16) float red[kConvWarps][32 * 8];
  const int CV = a.C / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cv = blockIdx.y * 32 + lane;
  const bool on = cv < CV;
  const int n_tiles = (a.N + TB - 1) / TB;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmDY);
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, status, limit_ns};
  float wr[K][8], dwl[K][8], dbl[8];
#pragma unroll
  for (int k = 0; k < K; ++k) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      dwl[k][e] = 0.f;
      wr[k][e] = 0.f;
    }
    if (on) load_w8(w + (size_t)k * a.C + 8 * cv, wr[k]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) dbl[e] = 0.f;
  auto issue = [&](int tl, int st) {
    mbar_expect_tx(&bars[st], 2 * BOX);           // two boxes land on this barrier
    tma_load_2d(smem + st * STAGE, &tmX, &bars[st], blockIdx.y * 256, tl * TB - (K - 1));
    tma_load_2d(smem + st * STAGE + HALF, &tmDY, &bars[st], blockIdx.y * 256, tl * TB);
  };
  int tile = blockIdx.x;
  if (threadIdx.x == 0 && tile < n_tiles) issue(tile, 0);
  if (tile < n_tiles) stage_ids(a, tile * TB - (K - 1), NIDS, ids[0]);
  cp_async_commit();
  int i = 0;
  bool aborted = false;
  for (; tile < n_tiles; ++i, tile += gridDim.x) {
    const int s = i & 1;
    const int next = tile + gridDim.x;
    if (next < n_tiles) {
      if (threadIdx.x == 0) issue(next, s ^ 1);
      stage_ids(a, next * TB - (K - 1), NIDS, ids[s ^ 1]);
    }
    cp_async_commit();
    cp_async_wait_prev();
    const bool ok = mbar_wait(&bars[s], (i >> 1) & 1, wc);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const uint8_t* xs = smem + s * STAGE + lane * 16;
    const uint8_t* ds = xs + HALF;
    const int T0 = tile * TB;
    if (on) {
#pragma unroll 2
      for (int r = warp; r < TB; r += kConvWarps) {
        const int t = T0 + r;
        if (t >= a.N) break;
        const int* id = ids[s] + r;               // id[K-1] is t's node; id[K-1-k] token t-k, id[K-1+k] t+k
        const int v = id[K - 1];
        float g[8], xv[8], acc[8];
        load8(reinterpret_cast<const uint4*>(ds + r * rs), g);
#pragma unroll
        for (int e = 0; e < 8; ++e) dbl[e] += g[e];
        // dw (and, for the first K-1 tokens of a node, the terms that cross into an ancestor)
        if (id[0] == v) {
#pragma unroll
          for (int k = 0; k < K; ++k) {
            load8(reinterpret_cast<const uint4*>(xs + (r + K - 1 - k) * rs), xv);
            fma8(dwl[k], xv, g);
          }
        } else {
          int off = 0;                            // tokens of v before t (< K-1 here)
          while (off < K - 1 && id[K - 2 - off] == v) ++off;
          int j = t;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            if (j < 0) break;
            load8(x + (size_t)j * CV + cv, xv);
            fma8(dwl[k], xv, g);
            if (k > off) {
              float c[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) c[e] = wr[k][e] * g[e];
              red_add8(ws + (size_t)j * a.C + 8 * cv, c);
            }
            j = path_prev1(j, a.tok_node, a.tok_start, a.parent, a.node_len, a.n_nodes);
          }
        }
        // dx: the successors inside the node, all staged (t + k < node end <= N)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = wr[0][e] * g[e];
        if (id[2 * (K - 1)] == v) {               // t .. t+K-1 all in t's node
#pragma unroll
          for (int k = 1; k < K; ++k) {
            load8(reinterpret_cast<const uint4*>(ds + (r + k) * rs), xv);
            fma8(acc, wr[k], xv);
          }
          dx[(size_t)t * CV + cv] = pack8(acc);
        } else {
#pragma unroll
          for (int k = 1; k < K; ++k) {
            if (id[K - 1 + k] != v) break;          // t+k past the node's end
            load8(reinterpret_cast<const uint4*>(ds + (r + k) * rs), xv);
            fma8(acc, wr[k], xv);
          }
          red_add8(ws + (size_t)t * a.C + 8 * cv, acc);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait_all();
  if (aborted) {
    if (threadIdx.x == 0) {
      drain_bar(&bars[i & 1], (i >> 1) & 1, limit_ns);
      if (tile + gridDim.x < n_tiles) drain_bar(&bars[(i & 1) ^ 1], ((i + 1) >> 1) & 1, limit_ns);
    }
    return;                                      // every thread leaves here: the reduction below is skipped
  }
  // block reduction of dw and db over the warps; 64 threads then add 4 floats each
  const int c4 = threadIdx.x;                    // float4 column of the block's 32 x 8 channels
  const int cv4 = blockIdx.y * 32 + (c4 >> 1);
#pragma unroll
  for (int k = 0; k <= K; ++k) {
    const float(&src)[8] = k < K ? dwl[k] : dbl;
    *reinterpret_cast<float4*>(&red[warp][lane * 8]) = make_float4(src[0], src[1], src[2], src[3]);
    *reinterpret_cast<float4*>(&red[warp][lane * 8 + 4]) = make_float4(src[4], src[5], src[6], src[7]);
    __syncthreads();
    if (c4 < 64 && cv4 < CV) {
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kConvWarps; ++q) {
        const float4 p = *reinterpret_cast<const float4*>(&red[q][c4 * 4]);
        sum.x += p.x; sum.y += p.y; sum.z += p.z; sum.w += p.w;
      }
      float* dst = k < K ? dw + (size_t)k * a.C : dbias;
      if (dst)
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 8 * cv4 + (c4 & 1) * 4), "f"(sum.x),
                     "f"(sum.y), "f"(sum.z), "f"(sum.w)
                     : "memory");
    }
    __syncthreads();
  }
}

// The boundary rows of node v: its last min(len, K-1) tokens.  Zeroed before k_conv_bwd (and dw,
// dbias by block (0, 0)), converted to bf16 after it.  Blocks over nodes (x, grid-stride) and
// chunks of the rows' channels (y).
__global__ void __launch_bounds__(256) k_conv_bwd_zero(ConvArgs a, float* ws, float* dw, float* dbias) {
  const int C4 = a.C / 4;
  const int i0 = blockIdx.y * blockDim.x + threadIdx.x, step = gridDim.y * blockDim.x;
  if (blockIdx.x == 0) {
    for (int i = i0; i < a.K * C4; i += step) reinterpret_cast<float4*>(dw)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (dbias)
      for (int i = i0; i < C4; i += step) reinterpret_cast<float4*>(dbias)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int v = blockIdx.x; v < a.n_nodes; v += gridDim.x) {
    const int len = a.node_len[v];
    const int rows = min(len, a.K - 1);
    const size_t r0 = (size_t)(a.tok_start[v] + len - rows);
    for (int i = i0; i < rows * C4; i += step)
      reinterpret_cast<float4*>(ws + r0 * a.C)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__global__ void __launch_bounds__(256) k_conv_bwd_finish(ConvArgs a, const float* __restrict__ ws,
                                                         uint2* __restrict__ dx) {
  const int C4 = a.C / 4;
  const int i0 = blockIdx.y * blockDim.x + threadIdx.x, step = gridDim.y * blockDim.x;
  for (int v = blockIdx.x; v < a.n_nodes; v += gridDim.x) {
    const int len = a.node_len[v];
    const int rows = min(len, a.K - 1);
    const size_t r0 = (size_t)(a.tok_start[v] + len - rows);
    for (int i = i0; i < rows * C4; i += step) {
      const float4 f = reinterpret_cast<const float4*>(ws + r0 * a.C)[i];
      dx[r0 * C4 + i] = make_uint2(pack_bf16(f.x, f.y), pack_bf16(f.z, f.w));
    }
  }
}

// state routing: one thread per (node, 4 state floats)
__global__ void k_route_fwd(const int32_t* __restrict__ parent, const int32_t* __restrict__ node_len, int n, int S4,
                            const float4* __restrict__ fin, float4* init) {
  const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= (size_t)n * S4) return;
  const int v = static_cast<int>(g / S4), s = static_cast<int>(g % S4);
  const int a = token_ancestor(v, parent, node_len, n);
  init[g] = a < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : fin[(size_t)a * S4 + s];
}

__global__ void k_route_bwd(const int32_t* __restrict__ parent, const int32_t* __restrict__ node_len, int n, int S4,
                            const float4* __restrict__ d_init, float* d_fin) {
  const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= (size_t)n * S4) return;
  const int v = static_cast<int>(g / S4), s = static_cast<int>(g % S4);
  const int a = token_ancestor(v, parent, node_len, n);
  if (a < 0) return;
  const float4 d = d_init[g];
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(d_fin + ((size_t)a * S4 + s) * 4), "f"(d.x),
               "f"(d.y), "f"(d.z), "f"(d.w)
               : "memory");
}

int conv_args(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len, int C, int K, ConvArgs* a) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!parent || !node_len) return TREE_ERR_ARG;
  if (C <= 0 || C % 8 != 0 || K < 1 || K > kConvMaxK) return TREE_ERR_SHAPE;
  *a = ConvArgs{plan->tok_node, plan->tok_start, parent, node_len, plan->n_tokens, C, K, plan->n_nodes};
  return TREE_OK;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

// channels per staged row: a 256-channel slab, or all C when fewer
int conv_box(int C) { return std::min(C, 256); }

// Persistent grid: as many blocks as fit on the GPU at once, split over the channel slabs;
// each block then walks its share of the token tiles.
template <typename Kern>
int conv_grid(Kern kern, int smem_bytes, int n_tiles, int slabs, dim3* grid) {
  int rc = record_cuda(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes));
  if (rc) return rc;
  int dev = 0, sms = 0, per_sm = 0;
  rc = record_cuda(cudaGetDevice(&dev));
  if (!rc) rc = record_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (!rc) rc = record_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem_bytes));
  if (rc) return rc;
  const int resident = std::max(1, per_sm) * sms;
  *grid = dim3((unsigned)std::max(1, std::min(n_tiles, resident / slabs)), (unsigned)slabs);
  return TREE_OK;
}

template <int K>
int launch_conv_fwd(const CUtensorMap& tx, const ConvArgs& a, const tree_bf16* x, const float* w, const float* bias,
                    tree_bf16* y, int32_t* status, cudaStream_t s) {
  constexpr int smem = 2 * (kConvFwdTile + K - 1) * kConvRowBytes + 1024;
  dim3 grid;
  int rc = conv_grid(k_conv_fwd<K>, smem, (a.N + kConvFwdTile - 1) / kConvFwdTile, (a.C / 8 + 31) / 32, &grid);
  if (rc) return rc;
  k_conv_fwd<K><<<grid, 256, smem, s>>>(tx, a, reinterpret_cast<const uint4*>(x), w, bias,
                                         reinterpret_cast<uint4*>(y), conv_box(a.C) * 2, status, wait_limit_ns());
  return record_cuda(cudaGetLastError());
}

template <int K>
int launch_conv_bwd(const CUtensorMap& tx, const CUtensorMap& tdy, const ConvArgs& a, const tree_bf16* x,
                    const float* w, float* ws, tree_bf16* dx, float* dw, float* dbias, int32_t* status,
                    cudaStream_t s) {
  constexpr int smem = 4 * (kConvBwdTile + K - 1) * kConvRowBytes + 1024;
  dim3 grid;
  int rc = conv_grid(k_conv_bwd<K>, smem, (a.N + kConvBwdTile - 1) / kConvBwdTile, (a.C / 8 + 31) / 32, &grid);
  if (rc) return rc;
  k_conv_bwd<K><<<grid, 256, smem, s>>>(tx, tdy, a, reinterpret_cast<const uint4*>(x), w, ws,
                                         reinterpret_cast<uint4*>(dx), dw, dbias, conv_box(a.C) * 2, status,
                                         wait_limit_ns());
  return record_cuda(cudaGetLastError());
}

}  // namespace
}  // namespace ta

using namespace ta;

extern "C" {

int tree_conv1d_fwd(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len, const tree_bf16* x,
                    const float* w, const float* bias, int C, int K, tree_bf16* y, int32_t* status_dev,
                    tree_stream_t stream) {
  ConvArgs a;
  int rc = conv_args(plan, parent, node_len, C, K, &a);
  if (rc) return rc;
  if (!x || !w || !y || misaligned(x) || misaligned(w) || misaligned(y) || (bias && misaligned(bias)))
    return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  CUtensorMap tx;
  rc = make_tmap_bf16_2d(&tx, x, C, a.N, conv_box(C), kConvFwdTile + K - 1);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (K) {
#define TA_CONV_FWD(KK) \
  case KK: return launch_conv_fwd<KK>(tx, a, x, w, bias, y, status_dev, s);
    TA_CONV_FWD(1) TA_CONV_FWD(2) TA_CONV_FWD(3) TA_CONV_FWD(4)
    TA_CONV_FWD(5) TA_CONV_FWD(6) TA_CONV_FWD(7) TA_CONV_FWD(8)
#undef TA_CONV_FWD
  }
  return TREE_ERR_SHAPE;
}

size_t tree_conv1d_bwd_workspace(const tree_plan_t* plan, int C) {
  if (!plan || C <= 0) return 0;
  return (size_t)plan->n_tokens * C * 4;
}

int tree_conv1d_bwd(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len, const tree_bf16* x,
                    const float* w, const tree_bf16* dy, int C, int K, void* workspace, tree_bf16* dx, float* dw,
                    float* dbias, int32_t* status_dev, tree_stream_t stream) {
  ConvArgs a;
  int rc = conv_args(plan, parent, node_len, C, K, &a);
  if (rc) return rc;
  if (!x || !w || !dy || !workspace || !dx || !dw)
    return TREE_ERR_ARG;
  for (const void* p : {(const void*)x, (const void*)w, (const void*)dy, (const void*)workspace, (const void*)dx,
                        (const void*)dw})
    if (misaligned(p)) return TREE_ERR_ARG;
  if (dbias && misaligned(dbias)) return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  CUtensorMap tx, tdy;
  rc = make_tmap_bf16_2d(&tx, x, C, a.N, conv_box(C), kConvBwdTile + K - 1);
  if (!rc) rc = make_tmap_bf16_2d(&tdy, dy, C, a.N, conv_box(C), kConvBwdTile + K - 1);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  const int row_chunks = std::max(1, std::min(16, ((std::max(K - 1, 1)) * (C / 4) + 255) / 256));
  const dim3 node_blocks((unsigned)std::max(1, std::min(a.n_nodes, 152 * 8)), (unsigned)row_chunks);
  k_conv_bwd_zero<<<node_blocks, 256, 0, s>>>(a, ws, dw, dbias);
  rc = record_cuda(cudaGetLastError());
  if (rc) return rc;
  switch (K) {
#define TA_CONV_BWD(KK) \
  case KK: rc = launch_conv_bwd<KK>(tx, tdy, a, x, w, ws, dx, dw, dbias, status_dev, s); break;
    TA_CONV_BWD(1) TA_CONV_BWD(2) TA_CONV_BWD(3) TA_CONV_BWD(4)
    TA_CONV_BWD(5) TA_CONV_BWD(6) TA_CONV_BWD(7) TA_CONV_BWD(8)
#undef TA_CONV_BWD
  }
  if (rc) return rc;
  if (K > 1) k_conv_bwd_finish<<<node_blocks, 256, 0, s>>>(a, ws, reinterpret_cast<uint2*>(dx));
  return record_cuda(cudaGetLastError());
}

int tree_route_states(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, const float* final_states,
                      int S, float* init_states, tree_stream_t stream) {
  if (!parent || !node_len || !final_states || !init_states || n_nodes <= 0) return TREE_ERR_ARG;
  if (S <= 0 || S % 4 != 0) return TREE_ERR_SHAPE;
  if (misaligned(final_states) || misaligned(init_states)) return TREE_ERR_ARG;
  int rc = check_device();
  if (rc) return rc;
  const size_t items = (size_t)n_nodes * (S / 4);
  k_route_fwd<<<(unsigned)((items + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      parent, node_len, n_nodes, S / 4, reinterpret_cast<const float4*>(final_states),
      reinterpret_cast<float4*>(init_states));
  return record_cuda(cudaGetLastError());
}

int tree_route_states_bwd(const int32_t* parent, const int32_t* node_len, int32_t n_nodes, const float* d_init,
                          int S, float* d_final, tree_stream_t stream) {
  if (!parent || !node_len || !d_init || !d_final || n_nodes <= 0) return TREE_ERR_ARG;
  if (S <= 0 || S % 4 != 0) return TREE_ERR_SHAPE;
  if (misaligned(d_init) || misaligned(d_final)) return TREE_ERR_ARG;
  int rc = check_device();
  if (rc) return rc;
  const size_t items = (size_t)n_nodes * (S / 4);
  k_route_bwd<<<(unsigned)((items + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      parent, node_len, n_nodes, S / 4, reinterpret_cast<const float4*>(d_init), d_final);
  return record_cuda(cudaGetLastError());
}

}  // extern "C"
