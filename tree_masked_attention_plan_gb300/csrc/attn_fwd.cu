// Tree-masked attention forward on tcgen05 ("Tree Training 技术详解", section 4.2:
// Softmax(Q K^T / sqrt(d) + M) V with the tree mask M; section 4.3: block-sparse over the
// ancestor tiles, mask evaluated only where a tile is partly visible).
//
// One CTA computes one (query tile, q head) pair over the non-empty key tiles of its row:
//   warp 0      TMA producer: Q tile once, then K/V tiles (plus their dfs_in/dfs_out words)
//               into a 2-stage ring;
//   warp 1      allocates TMEM and issues every tcgen05.mma from one thread:
//               S_b = Q K^T into one of two TMEM score buffers, O += P V into the TMEM
//               output accumulator;
//   warps 2..5  softmax: thread r owns query row r (TMEM lane r), so the running max and
//               sum of a row stay in that thread; partial tiles apply the interval mask
//               dfs_in(node j) <= dfs_in(node i) <= dfs_out(node j) and j <= i; P goes to
//               shared memory as bf16 in the 128-byte-swizzled K-major layout the MMA reads;
//               O is rescaled in TMEM when the row max grows.
// Online-softmax state per row is (m, l) in log2 units; two partial states combine with
// the associative merge of the Tree Attention page (max of maxima, rescaled sums).
#include <cmath>

#include "common.cuh"

namespace ta {
namespace {

template <int HD>
struct FwdCfg {
  static constexpr int NCH = HD / 64;                 // 64-column (128-byte) chunks per row
  static constexpr int NS = 2;                        // K/V ring stages
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NCH * CHUNK_BYTES;
  static constexpr int V_OFF = K_OFF + NS * NCH * CHUNK_BYTES;
  static constexpr int P_OFF = V_OFF + NS * NCH * CHUNK_BYTES;
  static constexpr int KIN_OFF = P_OFF + 2 * CHUNK_BYTES;
  static constexpr int KOUT_OFF = KIN_OFF + NS * TILE * 4;
  static constexpr int BAR_OFF = KOUT_OFF + NS * TILE * 4;
  static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 1 + 1 + 1;   // q, kv full/empty, s full/free, p, pv, drain
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;      // slack for 1024-byte alignment
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 256;
  static constexpr uint32_t IDESC_S = idesc_bf16(TILE, TILE, 0, 0);   // Q K-major, K K-major
  static constexpr uint32_t IDESC_PV = idesc_bf16(TILE, HD, 0, 1);    // P K-major, V MN-major
  static constexpr uint32_t KV_TX = 2 * NCH * CHUNK_BYTES + 2 * TILE * 4;
};

struct FwdParams {
  const int32_t* row_ptr;
  const int32_t* row_idx;
  const int32_t* row_order;
  const int32_t* tok_in;
  const int32_t* tok_out;
  const uint8_t* tile_class;
  __nv_bfloat16* o;
  float* lse;
  int32_t* status;
  int N, T, Npad, Hq, grp;
  float scale_log2;          // softmax scale * log2(e)
  uint64_t wait_ns;
};

constexpr int kFwdThreads = 192;

DEVI uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// Time-bounded wait that ignores the abort flag (used to drain in-flight async work).
DEVI void mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return;
}

template <int HD>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + C::NS;
  uint64_t* s_full = bars + 1 + 2 * C::NS;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  int* abort_flag = reinterpret_cast<int*>(sm + C::MISC_OFF + 4);
  int32_t* kin_s = reinterpret_cast<int32_t*>(sm + C::KIN_OFF);
  int32_t* kout_s = reinterpret_cast<int32_t*>(sm + C::KOUT_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int qt = p.row_order[u / p.Hq];
  const int h = u % p.Hq;
  const int kvh = h / p.grp;
  const int rp0 = p.row_ptr[qt];
  const int cnt = p.row_ptr[qt + 1] - rp0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) { mbar_init(&kv_full[s], 1); mbar_init(&kv_empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&s_full[b], 1); mbar_init(&s_free[b], 128); }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.wait_ns};

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_expect_tx(q_full, C::NCH * CHUNK_BYTES);
      for (int c = 0; c < C::NCH; ++c) tma_load_3d(sm + C::Q_OFF + c * CHUNK_BYTES, &tmQ, q_full, c * 64, h, qt * TILE);
      int issued = 0;
      for (int n = 0; n < cnt; ++n) {
        const int s = n % C::NS;
        if (n >= C::NS && !mbar_wait(&kv_empty[s], ((n / C::NS) - 1) & 1, wc)) break;
        const int kt = p.row_idx[rp0 + n];
        mbar_expect_tx(&kv_full[s], C::KV_TX);
        uint8_t* kb = sm + C::K_OFF + s * C::NCH * CHUNK_BYTES;
        uint8_t* vb = sm + C::V_OFF + s * C::NCH * CHUNK_BYTES;
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(kb + c * CHUNK_BYTES, &tmK, &kv_full[s], c * 64, kvh, kt * TILE);
          tma_load_3d(vb + c * CHUNK_BYTES, &tmV, &kv_full[s], c * 64, kvh, kt * TILE);
        }
        bulk_load(kin_s + s * TILE, p.tok_in + (size_t)kt * TILE, TILE * 4, &kv_full[s]);
        bulk_load(kout_s + s * TILE, p.tok_out + (size_t)kt * TILE, TILE * 4, &kv_full[s]);
        issued = n + 1;
      }
      if (*abort_flag) {                       // let copies in flight land before exit
        mbar_wait_drain(q_full, 0, p.wait_ns);
        for (int n = (issued > C::NS ? issued - C::NS : 0); n < issued; ++n)
          mbar_wait_drain(&kv_full[n % C::NS], (n / C::NS) & 1, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(sm + C::Q_OFF);
      const uint32_t p_base = smem_u32(sm + C::P_OFF);
      auto issue_pv = [&](int m) -> bool {
        const int s = m % C::NS;
        if (!mbar_wait(p_full, m & 1, wc)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sm + C::V_OFF + s * C::NCH * CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;   // P: K-major, keys along K
          const uint32_t b_off = kk * 16 * 128;                             // V: 16 key rows per step
          umma_bf16(tmem + C::O_COL, sdesc_sw128(p_base + a_off, 16, 1024),
                    sdesc_sw128(v_base + b_off, CHUNK_BYTES, 1024), C::IDESC_PV, (m > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&kv_empty[s]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, wc);
      for (int n = 0; ok && n < cnt; ++n) {
        const int s = n % C::NS, b = n & 1;
        if (!mbar_wait(&kv_full[s], (n / C::NS) & 1, wc)) { ok = false; break; }
        if (n >= 2 && !mbar_wait(&s_free[b], ((n >> 1) - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_base = smem_u32(sm + C::K_OFF + s * C::NCH * CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;     // d along K, 32 B per step
          umma_bf16(tmem + b * TILE, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024),
                    C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        if (n >= 1 && !issue_pv(n - 1)) { ok = false; break; }
      }
      if (ok && cnt > 0) issue_pv(cnt - 1);
      umma_commit(drain);                      // completes once every MMA above is done
      mbar_wait_drain(drain, 0, p.wait_ns);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int wq = warp & 3;                   // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;              // query row inside the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const int qi = qt * TILE + r;
    const int qin = p.tok_in[qi];
    float m_run = -INFINITY;                   // running row max (log2 units)
    float m_ref = 0.f;                         // offset the current O and l are scaled by
    float l_run = 0.f;
    bool ok = true;
    for (int n = 0; n < cnt; ++n) {
      const int b = n & 1, s = n % C::NS;
      const int kt = p.row_idx[rp0 + n];
      const uint8_t cls = p.tile_class[(size_t)qt * p.T + kt];
      if (!mbar_wait_warp(&s_full[b], (n >> 1) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      float sv[TILE];
#pragma unroll
      for (int j = 0; j < TILE / 32; ++j) {
        uint32_t rr[32];
        tmem_load32(lane_base + b * TILE + j * 32, rr);
#pragma unroll
        for (int c = 0; c < 32; ++c) sv[j * 32 + c] = __uint_as_float(rr[c]);
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      if (cls == 1) {                          // partial tile: tree mask in registers
        if (!mbar_wait_warp(&kv_full[s], (n / C::NS) & 1, wc)) { ok = false; break; }
        const int4* kin4 = reinterpret_cast<const int4*>(kin_s + s * TILE);
        const int4* kout4 = reinterpret_cast<const int4*>(kout_s + s * TILE);
        const int jrel = qi - kt * TILE;       // key c is causal-visible iff c <= jrel
#pragma unroll
        for (int c4 = 0; c4 < TILE / 4; ++c4) {
          const int4 a = kin4[c4], z = kout4[c4];
          const int c = c4 * 4;
          if (!(c + 0 <= jrel && a.x <= qin && qin <= z.x)) sv[c + 0] = -INFINITY;
          if (!(c + 1 <= jrel && a.y <= qin && qin <= z.y)) sv[c + 1] = -INFINITY;
          if (!(c + 2 <= jrel && a.z <= qin && qin <= z.z)) sv[c + 2] = -INFINITY;
          if (!(c + 3 <= jrel && a.w <= qin && qin <= z.w)) sv[c + 3] = -INFINITY;
        }
      }
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = sv[e];
#pragma unroll
      for (int c = 8; c < TILE; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m_run, mt * p.scale_log2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (l_run == 0.f) ? 0.f : ex2_approx(m_ref - m_use);
      uint32_t pk[TILE / 2];
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < TILE; c += 2) {
        const float p0 = ex2_approx(fmaf(sv[c], p.scale_log2, -m_use));
        const float p1 = ex2_approx(fmaf(sv[c + 1], p.scale_log2, -m_use));
        rs[(c >> 1) & 3] += p0 + p1;
        pk[c >> 1] = pack_bf16(p0, p1);
      }
      l_run = l_run * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
      if (n > 0) {
        if (!mbar_wait_warp(pv_done, (n - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        // TMEM ld/st are warp-collective: rescale when any row of the warp needs it
        // (rows whose max did not move have alpha == 1 and are multiplied exactly by 1)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int j = 0; j < HD / 32; ++j) {
            uint32_t rr[32];
            tmem_load32(lane_base + C::O_COL + j * 32, rr);
#pragma unroll
            for (int c = 0; c < 32; ++c) rr[c] = __float_as_uint(__uint_as_float(rr[c]) * alpha);
            tmem_store32(lane_base + C::O_COL + j * 32, rr);
          }
          tmem_wait_st();
        }
      }
      uint8_t* pbox = sm + C::P_OFF;
#pragma unroll
      for (int uu = 0; uu < TILE / 8; ++uu)
        st_swizzled_unit(pbox + (uu >> 3) * CHUNK_BYTES, r, uu & 7,
                         make_uint4(pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]));
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      m_run = m_new;
      m_ref = m_use;
    }
    if (ok && cnt > 0 && mbar_wait_warp(pv_done, (cnt - 1) & 1, wc)) {
      tc_fence_after();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow = p.o + ((size_t)qi * p.Hq + h) * HD;
#pragma unroll
      for (int j = 0; j < HD / 32; ++j) {
        uint32_t rr[32];
        tmem_load32(lane_base + C::O_COL + j * 32, rr);
        if (qi < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + j * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int c = v * 8;
            dst[v] = make_uint4(
                pack_bf16(__uint_as_float(rr[c + 0]) * inv_l, __uint_as_float(rr[c + 1]) * inv_l),
                pack_bf16(__uint_as_float(rr[c + 2]) * inv_l, __uint_as_float(rr[c + 3]) * inv_l),
                pack_bf16(__uint_as_float(rr[c + 4]) * inv_l, __uint_as_float(rr[c + 5]) * inv_l),
                pack_bf16(__uint_as_float(rr[c + 6]) * inv_l, __uint_as_float(rr[c + 7]) * inv_l));
          }
        }
      }
      p.lse[(size_t)h * p.Npad + qi] = (qi < p.N && l_run > 0.f) ? (m_ref + log2f(l_run)) * 0.69314718055994531f : 0.f;
    }
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int HD>
int launch_fwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, const tree_bf16* v, int Hq,
               int Hkv, float scale, tree_bf16* o, float* lse, int32_t* status, cudaStream_t s) {
  using C = FwdCfg<HD>;
  const int N = plan->n_tokens, T = plan->n_tiles;
  CUtensorMap tq, tk, tv;
  int rc = make_tmap_bf16_3d(&tq, q, HD, Hq, N);
  if (!rc) rc = make_tmap_bf16_3d(&tk, k, HD, Hkv, N);
  if (!rc) rc = make_tmap_bf16_3d(&tv, v, HD, Hkv, N);
  if (rc) return rc;
  rc = record_cuda(cudaFuncSetAttribute(k_attn_fwd<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC));
  if (rc) return rc;
  FwdParams P{plan->row_ptr, plan->row_idx, plan->row_order, plan->tok_in, plan->tok_out, plan->tile_class,
              reinterpret_cast<__nv_bfloat16*>(o), lse, status, N, T, T * TILE, Hq, Hq / Hkv,
              scale * 1.4426950408889634f, wait_limit_ns()};
  k_attn_fwd<HD><<<T * Hq, kFwdThreads, C::SMEM_ALLOC, s>>>(tq, tk, tv, P);
  return record_cuda(cudaGetLastError());
}

}  // namespace
}  // namespace ta

using namespace ta;

extern "C" int tree_attn_fwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, const tree_bf16* v,
                             int Hq, int Hkv, int d, float scale, tree_bf16* o, float* lse, int32_t* status_dev,
                             tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse) return TREE_ERR_ARG;
  if ((d != 64 && d != 128) || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return TREE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(o) & 15) || (reinterpret_cast<uintptr_t>(lse) & 3)) return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  if (!(scale > 0.f)) scale = 1.f / sqrtf(static_cast<float>(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 128 ? launch_fwd<128>(plan, q, k, v, Hq, Hkv, scale, o, lse, status_dev, s)
                  : launch_fwd<64>(plan, q, k, v, Hq, Hkv, scale, o, lse, status_dev, s);
}
