// Path-averaged next-token cross-entropy over the packed tree ("Tree Training 技术详解",
// sections 6.2, 6.3, 12), fused with the vocabulary projection and computed chunk by chunk
// so that only one chunk of logits gradients is ever materialised (the chunked, recomputed
// logits of the agent-RL tutorial, chapter 14 "规模扩展与效率", section 14.3).
//
// Pairs: token u (label not ignored) is predicted by the logits row of prev(u), the token
// before u on its root path (u-1 inside a node, the parent's last token for a node's first
// token), with weight c_u = g_u / K.  Per logits row t:
//   loss   += sum_{u: prev(u)=t} c_u (LSE_t - z_t[y_u]),     z_t = W h_t
//   dz_t    = csum_t softmax(z_t) - sum_{u: prev(u)=t} c_u e_{y_u},   csum_t = sum c_u
//   dh_t    = dz_t W,     dW += dz^T h.
// Per chunk of rows: (1) logits GEMM whose epilogue keeps each row's (max, sum exp) per
// 256-column tile, (2) merge to LSE, (3) the logits GEMM again whose epilogue writes
// dz = csum softmax in bf16, (4) the -c_u at the labels, (5) dh = dz W, (6) dW += dz^T h.
// All four products run on one tcgen05 GEMM kernel: 128 x 256 output tile per CTA, fp32
// accumulator in TMEM, 64-deep K stages of bf16 operands brought in by TMA with the 128-byte
// swizzle, either operand K-major or MN-major (so that dz serves both as dz and as dz^T and
// W as W^T without transposed copies).
#include <algorithm>

#include <cuda_bf16.h>

#include "common.cuh"

namespace ta {
int make_tmap_bf16_2d_sw128(CUtensorMap* m, const void* base, int inner, int rows, int box_inner,
                            int box_rows);  // host.cu

namespace {

constexpr int GM = 128, GN = 256, GK = 64;         // CTA tile and K per stage
constexpr int GSTAGES = 2;                         // two CTAs per SM: four stages in flight
constexpr int A_BYTES = GM * GK * 2;               // 16 KB
constexpr int B_BYTES = GN * GK * 2;               // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MN_BOX_BYTES = 64 * GK * 2;          // one 64-wide MN block of 64 K rows: 8 KB
constexpr int G_BAR_OFF = GSTAGES * STAGE_BYTES;
constexpr int G_SMEM = G_BAR_OFF + (2 * GSTAGES + 1) * 8 + 16;
constexpr int G_SMEM_ALLOC = G_SMEM + 1024;        // slack for 1024-byte alignment
constexpr int G_THREADS = 192;                     // producer, MMA issuer, four epilogue warps
constexpr uint32_t G_TMEM_COLS = 256;
constexpr float kLog2e = 1.4426950408889634f;

enum Epi { EPI_LSE = 0, EPI_DZ = 1, EPI_BF16 = 2, EPI_F32 = 3 };

struct GemmArgs {
  int M, N, K;          // valid output rows and columns, contraction length
  int a_off, b_off;     // added to each operand's second TMA coordinate (rows of a K-major
                        // operand, K of an MN-major one)
  float2* part;         // EPI_LSE: [M][part_ld] (max, sum exp) per 256-column tile
  int part_ld;
  const float* lse;     // EPI_DZ: per output row
  const float* csum;
  __nv_bfloat16* out_bf16;   // EPI_DZ, EPI_BF16: row stride ld elements
  float* out_f32;            // EPI_F32: row stride ld; acc_first = 1 overwrites, else adds
  int ld, acc_first;
  int32_t* status;
  uint64_t limit_ns;
};

DEVI uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

DEVI void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

DEVI void drain_bar(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < limit_ns) {
  }
}

// C tile (blockIdx.x, blockIdx.y) = (m tile, n tile) for the logits products (consecutive
// CTAs share one vocabulary tile, the chunk's hidden states stay in L2) and (n tile, m tile)
// for dh and dW (consecutive CTAs share one row panel of dz).
template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(G_THREADS, 2) k_gemm(const __grid_constant__ CUtensorMap tmA,
                                                       const __grid_constant__ CUtensorMap tmB, const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + G_BAR_OFF);
  uint64_t* empty = full + GSTAGES;
  uint64_t* acc_full = empty + GSTAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr bool LOGITS = (EPI == EPI_LSE || EPI == EPI_DZ);
  const int mt = LOGITS ? blockIdx.x : blockIdx.y;
  const int nt = LOGITS ? blockIdx.y : blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (g.K + GK - 1) / GK;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < GSTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, G_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, g.status, g.limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % GSTAGES;
        if (kb >= GSTAGES && !mbar_wait(&empty[s], ((kb / GSTAGES) - 1) & 1, wc)) break;
        mbar_expect_tx(&full[s], STAGE_BYTES);
        uint8_t* a = sm + s * STAGE_BYTES;
        uint8_t* b = a + A_BYTES;
        const int k = kb * GK;
        if (A_MN) {
          tma_load_2d(a, &tmA, &full[s], mt * GM, g.a_off + k);
          tma_load_2d(a + MN_BOX_BYTES, &tmA, &full[s], mt * GM + 64, g.a_off + k);
        } else {
          tma_load_2d(a, &tmA, &full[s], k, g.a_off + mt * GM);
        }
        if (B_MN) {
#pragma unroll
          for (int j = 0; j < GN / 64; ++j)
            tma_load_2d(b + j * MN_BOX_BYTES, &tmB, &full[s], nt * GN + j * 64, g.b_off + k);
        } else {
          tma_load_2d(b, &tmB, &full[s], k, g.b_off + nt * GN);
        }
        issued = kb + 1;
      }
      if (*abort_flag)     // let the copies in flight land before the CTA's shared memory goes
        for (int kb = max(0, issued - GSTAGES); kb < issued; ++kb)
          drain_bar(&full[kb % GSTAGES], (kb / GSTAGES) & 1, g.limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(GM, GN, A_MN ? 1 : 0, B_MN ? 1 : 0);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % GSTAGES;
        if (!mbar_wait(&full[s], (kb / GSTAGES) & 1, wc)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(sm + s * STAGE_BYTES), b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < GK / 16; ++kk) {
          // K-major: 16 K elements = 32 bytes along the swizzled 128-byte row;
          // MN-major: 16 K rows of 128 bytes, 64-wide MN blocks 8 KB apart
          const uint64_t ad = A_MN ? sdesc_sw128(a + kk * 2048, MN_BOX_BYTES, 1024) : sdesc_sw128(a + kk * 32, 16, 1024);
          const uint64_t bd = B_MN ? sdesc_sw128(b + kk * 2048, MN_BOX_BYTES, 1024) : sdesc_sw128(b + kk * 32, 16, 1024);
          umma_bf16(tmem, ad, bd, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(acc_full);   // arrives once every MMA issued above has completed
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;                        // TMEM lanes 32q .. 32q+31
    const int row = q * 32 + lane;
    const int grow = mt * GM + row;                // output row
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool ok = mbar_wait_warp(acc_full, 0, wc);
    tc_fence_after();
    if (ok && !*abort_flag) {
      const bool live = grow < g.M;
      if (EPI == EPI_LSE) {
        float m = -INFINITY, ssum = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < GN; c0 += 32) {
          uint32_t r[32];
          tmem_load32(trow + c0, r);
          const int nvalid = min(32, g.N - (nt * GN + c0));
          float cm = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nvalid) cm = fmaxf(cm, __uint_as_float(r[i]));
          if (cm > m) {
            ssum *= ex2_approx((m - cm) * kLog2e);
            m = cm;
          }
          const float mb = m * kLog2e;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nvalid) ssum += ex2_approx(fmaf(__uint_as_float(r[i]), kLog2e, -mb));
        }
        if (live) g.part[(size_t)grow * g.part_ld + nt] = make_float2(m, ssum);
      } else if (EPI == EPI_DZ) {
        const float lb = live ? g.lse[grow] * kLog2e : 0.f;
        const float c = live ? g.csum[grow] : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < GN; c0 += 32) {
          uint32_t r[32];
          tmem_load32(trow + c0, r);
          const int col0 = nt * GN + c0;
          if (live && col0 < g.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16(c * ex2_approx(fmaf(__uint_as_float(r[2 * i]), kLog2e, -lb)),
                                c * ex2_approx(fmaf(__uint_as_float(r[2 * i + 1]), kLog2e, -lb)));
            uint4* dst = reinterpret_cast<uint4*>(g.out_bf16 + (size_t)grow * g.ld + col0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              if (col0 + 8 * v < g.N) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else if (EPI == EPI_BF16) {
#pragma unroll 1
        for (int c0 = 0; c0 < GN; c0 += 32) {
          uint32_t r[32];
          tmem_load32(trow + c0, r);
          const int col0 = nt * GN + c0;
          if (live && col0 < g.N) {
            uint4* dst = reinterpret_cast<uint4*>(g.out_bf16 + (size_t)grow * g.ld + col0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              if (col0 + 8 * v < g.N)
                dst[v] = make_uint4(pack_bf16(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1])),
                                    pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                    pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                    pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
          }
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < GN; c0 += 32) {
          uint32_t r[32];
          tmem_load32(trow + c0, r);
          const int col0 = nt * GN + c0;
          if (live && col0 < g.N) {
            float4* dst = reinterpret_cast<float4*>(g.out_f32 + (size_t)grow * g.ld + col0);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              if (col0 + 4 * v < g.N) {
                float4 o = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                       __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                if (!g.acc_first) {
                  const float4 p = dst[v];
                  o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
                }
                dst[v] = o;
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag && lane == 0) drain_bar(acc_full, 0, g.limit_ns);   // MMAs in flight finish first
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, G_TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Pairs, logsumexp merge, label terms, loss.

struct CeTree {
  const int32_t* tok_node;
  const int32_t* tok_start;
  const int32_t* parent;
  const int32_t* node_len;
  const float* w;           // g_t / K per token
  int N, n_nodes;
};

DEVI int ce_token_ancestor(int v, const CeTree& t) {
  int a = t.parent[v];
  for (int guard = 0; a >= 0 && a < t.n_nodes && t.node_len[a] == 0 && guard < t.n_nodes; ++guard) a = t.parent[a];
  return (a >= 0 && a < t.n_nodes && t.node_len[a] > 0) ? a : -1;
}

// pair_row[u] = prev(u) if u is supervised and has a predecessor, else -1; csum[prev(u)] += c_u
__global__ void k_ce_pairs(CeTree t, const int32_t* __restrict__ labels, int V, int ignore_index,
                           int32_t* pair_row, float* csum, int32_t* status) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= t.N) return;
  const int y = labels[u];
  int row = -1;
  if (y != ignore_index) {
    if (y < 0 || y >= V) {
      if (status) atomicExch(status, TREE_ERR_ARG);
    } else {
      const int v = t.tok_node[u];
      if (u > t.tok_start[v]) {
        row = u - 1;
      } else {
        const int a = ce_token_ancestor(v, t);
        row = a < 0 ? -1 : t.tok_start[a] + t.node_len[a] - 1;
      }
    }
  }
  pair_row[u] = row;
  if (row >= 0) atomicAdd(csum + row, t.w[u]);
}

// z_{prev(u)}[y_u] = h_{prev(u)} . W_{y_u} in fp32; a warp per token
__global__ void k_ce_label_logit(const int32_t* __restrict__ pair_row, const int32_t* __restrict__ labels,
                                 const uint4* __restrict__ h, const uint4* __restrict__ W, int N, int D, float* zl) {
  const int u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (u >= N) return;
  const int row = pair_row[u];
  if (row < 0) return;
  const int DV = D / 8;
  const uint4* hr = h + (size_t)row * DV;
  const uint4* wr = W + (size_t)labels[u] * DV;
  float acc = 0.f;
  for (int i = lane; i < DV; i += 32) {
    const uint4 a = hr[i], b = wr[i];
    acc = fmaf(bf16lo(a.x), bf16lo(b.x), acc); acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
    acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc); acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
    acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc); acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
    acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc); acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) zl[u] = acc;
}

// (m, s) <- the merge of two (max, sum exp) states; an empty state has m = -inf, s = 0
DEVI void merge_ms(float& m, float& s, float om, float os) {
  const float nm = fmaxf(m, om);
  if (nm == -INFINITY) return;
  s = (m == -INFINITY ? 0.f : s * ex2_approx((m - nm) * kLog2e)) +
      (om == -INFINITY ? 0.f : os * ex2_approx((om - nm) * kLog2e));
  m = nm;
}

// LSE of each row of the chunk from its tiles' (max, sum exp); a warp per row
__global__ void k_ce_lse(const float2* __restrict__ part, int nparts, int rows, float* lse) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (r >= rows) return;
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < nparts; i += 32) {
    const float2 p = part[(size_t)r * nparts + i];
    merge_ms(m, s, p.x, p.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
    merge_ms(m, s, om, os);
  }
  if (lane == 0) lse[r] = m + __logf(s);
}

// dz[prev(u) - r0][y_u] -= c_u for the pairs whose row lies in [r0, r0 + rows)
__global__ void k_ce_fix(const int32_t* __restrict__ pair_row, const int32_t* __restrict__ labels,
                         const float* __restrict__ w, int N, int r0, int rows, int V, __nv_bfloat16* dz) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= N) return;
  const int row = pair_row[u];
  if (row < r0 || row >= r0 + rows) return;
  atomicAdd(dz + (size_t)(row - r0) * V + labels[u], __float2bfloat16(-w[u]));
}

// loss = sum_u c_u (LSE_{prev(u)} - z_{prev(u)}[y_u]), accumulated in fp64
__global__ void k_ce_loss(const int32_t* __restrict__ pair_row, const float* __restrict__ w,
                          const float* __restrict__ lse, const float* __restrict__ zl, int N, double* acc) {
  __shared__ double red[8];
  double v = 0.0;
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < N; u += gridDim.x * blockDim.x) {
    const int row = pair_row[u];
    if (row >= 0) v += (double)w[u] * ((double)lse[row] - (double)zl[u]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    atomicAdd(acc, s);
  }
}

__global__ void k_ce_loss_out(const double* acc, float* loss) { *loss = static_cast<float>(*acc); }

// ---------------------------------------------------------------------------------------------
// host side

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct CeLayout {
  size_t pair_row, zl, csum, lse, part, dz, acc, total;
};

CeLayout ce_layout(int N, int V, int chunk) {
  CeLayout L{};
  const size_t nparts = (size_t)(V + GN - 1) / GN;
  size_t o = 0;
  L.pair_row = o; o = align256(o + (size_t)N * 4);
  L.zl = o;       o = align256(o + (size_t)N * 4);
  L.csum = o;     o = align256(o + (size_t)N * 4);
  L.lse = o;      o = align256(o + (size_t)N * 4);
  L.part = o;     o = align256(o + (size_t)chunk * nparts * 8);
  L.dz = o;       o = align256(o + (size_t)chunk * V * 2);
  L.acc = o;      o = align256(o + 8);
  L.total = o;
  return L;
}

template <bool A_MN, bool B_MN, int EPI>
int launch_gemm(const CUtensorMap& ta_, const CUtensorMap& tb_, const GemmArgs& g, cudaStream_t s) {
  auto kern = k_gemm<A_MN, B_MN, EPI>;
  int rc = record_cuda(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM_ALLOC));
  if (rc) return rc;
  const unsigned mtiles = (unsigned)((g.M + GM - 1) / GM), ntiles = (unsigned)((g.N + GN - 1) / GN);
  const bool logits = (EPI == EPI_LSE || EPI == EPI_DZ);
  const dim3 grid = logits ? dim3(mtiles, ntiles) : dim3(ntiles, mtiles);
  kern<<<grid, G_THREADS, G_SMEM_ALLOC, s>>>(ta_, tb_, g);
  return record_cuda(cudaGetLastError());
}

// Operand maps: a K-major operand [rows][K] gets box {64 (K), rows of the tile}; an MN-major
// operand [K][MN] gets box {64 (MN), 64 (K)}.
int map_kmajor(CUtensorMap* m, const void* base, int K, int rows, int tile_rows) {
  return make_tmap_bf16_2d_sw128(m, base, K, rows, GK, tile_rows);
}
int map_mnmajor(CUtensorMap* m, const void* base, int MN, int K) {
  return make_tmap_bf16_2d_sw128(m, base, MN, K, 64, GK);
}

}  // namespace
}  // namespace ta

using namespace ta;

extern "C" {

size_t tree_ce_workspace(const tree_plan_t* plan, int D, int V, int chunk) {
  if (!plan || D <= 0 || V <= 0 || chunk <= 0) return 0;
  const int rows = std::min(chunk, plan->n_tokens);
  return ce_layout(plan->n_tokens, V, rows).total;
}

int tree_ce_fwd_bwd(const tree_plan_t* plan, const int32_t* parent, const int32_t* node_len, const tree_bf16* h,
                    const tree_bf16* W, const int32_t* labels, int D, int V, int chunk, int ignore_index,
                    void* workspace, float* loss, float* lse_out, tree_bf16* dh, float* dW, int32_t* status_dev,
                    tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!parent || !node_len || !h || !W || !labels || !workspace || !loss || !dh || !dW) return TREE_ERR_ARG;
  if (D < GN || D % GN != 0 || V < 8 || V % 8 != 0 || chunk <= 0 || chunk % GM != 0) return TREE_ERR_SHAPE;
  for (const void* p : {(const void*)h, (const void*)W, (const void*)workspace, (const void*)dh, (const void*)dW})
    if (misaligned16(p)) return TREE_ERR_ARG;
  if (lse_out && misaligned16(lse_out)) return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int N = plan->n_tokens;
  const int crows = std::min(chunk, N);
  const CeLayout L = ce_layout(N, V, crows);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* pair_row = reinterpret_cast<int32_t*>(ws + L.pair_row);
  float* zl = reinterpret_cast<float*>(ws + L.zl);
  float* csum = reinterpret_cast<float*>(ws + L.csum);
  float* lse = lse_out ? lse_out : reinterpret_cast<float*>(ws + L.lse);
  float2* part = reinterpret_cast<float2*>(ws + L.part);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(ws + L.dz);
  double* acc = reinterpret_cast<double*>(ws + L.acc);
  const int nparts = (V + GN - 1) / GN;

  rc = record_cuda(cudaMemsetAsync(csum, 0, (size_t)N * 4, s));
  if (!rc) rc = record_cuda(cudaMemsetAsync(acc, 0, 8, s));
  if (rc) return rc;
  const CeTree t{plan->tok_node, plan->tok_start, parent, node_len, plan->w, N, plan->n_nodes};
  k_ce_pairs<<<(N + 255) / 256, 256, 0, s>>>(t, labels, V, ignore_index, pair_row, csum, status_dev);
  k_ce_label_logit<<<(N + 7) / 8, 256, 0, s>>>(pair_row, labels, reinterpret_cast<const uint4*>(h),
                                               reinterpret_cast<const uint4*>(W), N, D, zl);
  rc = record_cuda(cudaGetLastError());
  if (rc) return rc;

  // maps shared by the chunks
  CUtensorMap m_h_km, m_w_km, m_w_mn, m_h_mn;
  rc = map_kmajor(&m_h_km, h, D, N, GM);                       // logits A: h rows
  if (!rc) rc = map_kmajor(&m_w_km, W, D, V, GN);              // logits B: W rows
  if (!rc) rc = map_mnmajor(&m_w_mn, W, D, V);                 // dh B: W as [K = V][N = D]
  if (!rc) rc = map_mnmajor(&m_h_mn, h, D, N);                 // dW B: h as [K = tokens][N = D]
  if (rc) return rc;
  const uint64_t lim = wait_limit_ns();
  for (int r0 = 0; r0 < N; r0 += crows) {
    const int rows = std::min(crows, N - r0);
    CUtensorMap m_dz_km, m_dz_mn;
    rc = map_kmajor(&m_dz_km, dz, V, rows, GM);                // dh A: dz rows, K = V
    if (!rc) rc = map_mnmajor(&m_dz_mn, dz, V, rows);          // dW A: dz as [K = rows][M = V]
    if (rc) return rc;
    GemmArgs g{};
    g.status = status_dev;
    g.limit_ns = lim;
    // (1) logits -> per-tile (max, sum exp)
    g.M = rows; g.N = V; g.K = D; g.a_off = r0; g.b_off = 0;
    g.part = part; g.part_ld = nparts;
    rc = launch_gemm<false, false, EPI_LSE>(m_h_km, m_w_km, g, s);
    if (rc) return rc;
    // (2) LSE of the chunk's rows
    k_ce_lse<<<(rows + 7) / 8, 256, 0, s>>>(part, nparts, rows, lse + r0);
    // (3) logits again -> dz = csum softmax (bf16)
    g.lse = lse + r0; g.csum = csum + r0; g.out_bf16 = dz; g.ld = V;
    rc = launch_gemm<false, false, EPI_DZ>(m_h_km, m_w_km, g, s);
    if (rc) return rc;
    // (4) -c_u at the labels
    k_ce_fix<<<(N + 255) / 256, 256, 0, s>>>(pair_row, labels, plan->w, N, r0, rows, V, dz);
    // (5) dh rows = dz W
    GemmArgs g2{};
    g2.status = status_dev; g2.limit_ns = lim;
    g2.M = rows; g2.N = D; g2.K = V; g2.a_off = 0; g2.b_off = 0;
    g2.out_bf16 = reinterpret_cast<__nv_bfloat16*>(dh) + (size_t)r0 * D; g2.ld = D;
    rc = launch_gemm<false, true, EPI_BF16>(m_dz_km, m_w_mn, g2, s);
    if (rc) return rc;
    // (6) dW (+)= dz^T h
    GemmArgs g3{};
    g3.status = status_dev; g3.limit_ns = lim;
    g3.M = V; g3.N = D; g3.K = rows; g3.a_off = 0; g3.b_off = r0;
    g3.out_f32 = dW; g3.ld = D; g3.acc_first = r0 == 0;
    rc = launch_gemm<true, true, EPI_F32>(m_dz_mn, m_h_mn, g3, s);
    if (rc) return rc;
  }
  k_ce_loss<<<std::max(1, std::min((N + 255) / 256, 152 * 4)), 256, 0, s>>>(pair_row, plan->w, lse, zl, N, acc);
  k_ce_loss_out<<<1, 1, 0, s>>>(acc, loss);
  return record_cuda(cudaGetLastError());
}

// Diagnostic product C [M][N] fp32 = op(A) op(B)^T on the same GEMM kernel:
// a_mn = 0: A stored [M][K]; 1: A stored [K][M].  b_mn = 0: B stored [N][K]; 1: [K][N].
int tree_diag_gemm(const tree_bf16* A, const tree_bf16* B, int M, int N, int K, int a_mn, int b_mn, float* C,
                   int32_t* status_dev, tree_stream_t stream) {
  if (!A || !B || !C || misaligned16(A) || misaligned16(B) || misaligned16(C)) return TREE_ERR_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 8 || N % 8 || K % 8) return TREE_ERR_SHAPE;
  int rc = check_device();
  if (rc) return rc;
  CUtensorMap ma, mb;
  rc = a_mn ? map_mnmajor(&ma, A, M, K) : map_kmajor(&ma, A, K, M, GM);
  if (!rc) rc = b_mn ? map_mnmajor(&mb, B, N, K) : map_kmajor(&mb, B, K, N, GN);
  if (rc) return rc;
  GemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.out_f32 = C; g.ld = N; g.acc_first = 1;
  g.status = status_dev; g.limit_ns = wait_limit_ns();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!a_mn && !b_mn) return launch_gemm<false, false, EPI_F32>(ma, mb, g, s);
  if (!a_mn && b_mn) return launch_gemm<false, true, EPI_F32>(ma, mb, g, s);
  if (a_mn && !b_mn) return launch_gemm<true, false, EPI_F32>(ma, mb, g, s);
  return launch_gemm<true, true, EPI_F32>(ma, mb, g, s);
}

}  // extern "C"
