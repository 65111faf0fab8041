// Tree-masked attention backward on tcgen05 ("Tree Training 技术详解", section 6.2 and
// section 7: a shared ancestor's K/V receive the summed gradients of every descendant that
// sees them).  Three kernels:
//   k_bwd_pre      delta_i = sum_c dO_ic O_ic per (token, q head), stored as -delta scale with
//                  -LSE log2e beside it; zeroes the fp32 dQ accumulator on the way.
//   k_bwd_dkdv     one CTA per (key tile, kv head): loops over the q heads of the group and the
//                  non-empty query tiles of the key tile's column.  Per step, in TMEM:
//                    S^T  = K Q^T            (cols   0..127, lane = key)
//                    dP^T = V dO^T           (cols 128..255)
//                  the elementwise warps form P^T = exp2(S^T scale log2e - LSE log2e) (masked on
//                  partial tiles; packed bf16 back into cols 0..63) and dS^T = P^T (dP^T - delta)
//                  scale as bf16 in shared memory;
//                    dV  += P^T dO           (cols 256..256+d)     accumulated on chip,
//                    dK  += dS^T Q           (cols 256+d..256+2d)  written once at the end,
//                    dQ   = dS K             (cols 128..128+d, lane = query), added to the fp32
//                                            accumulator by TMA bulk reduce-adds of 8 KiB pieces
//                                            staged through shared memory.
//                  The steps are software-pipelined: the tensor core runs dQ, dK of step n-1,
//                  dP, dV of step n and S of step n+1 around the elementwise passes (P, then dS).
//                  dK gets the inverse RoPE rotation in the epilogue.
//   k_dq_finalize  dQ = R(pos)^T dQacc, fp32 -> bf16, token-major.
// The fp32 dQ accumulator keeps each (head, query tile) block contiguous ([d/4][128][4] per block),
// so the reductions of the CTAs working on one query tile touch one compact region of L2.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace ta {
namespace {

constexpr int kMaxList = 1024;      // column lists up to this length are staged in shared memory

template <int HD>
struct BwdCfg {
  static constexpr int NCH = HD / 64;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + NCH * CHUNK_BYTES;
  // Q is loaded twice per step: once for S^T = K Q^T (freed as soon as that product is done,
  // so the next step's copy has a whole step to arrive) and once for dK += dS^T Q
  static constexpr int Q_OFF = V_OFF + NCH * CHUNK_BYTES;     // [Q for S][Q for dK]
  static constexpr int DO_OFF = Q_OFF + 2 * NCH * CHUNK_BYTES;
  static constexpr int DST_OFF = DO_OFF + NCH * CHUNK_BYTES;
  // per step, in a ring of two stages: -LSE log2e, -delta scale, query dfs_in, node runs of the query tile
  static constexpr int AUX_LSE = 0, AUX_DLT = TILE * 4, AUX_QIN = 2 * TILE * 4, AUX_RUNS = 3 * TILE * 4;
  static constexpr int AUX_BYTES = AUX_RUNS + TREE_MAX_RUNS * 16;
  static constexpr int AUX_OFF = DST_OFF + 2 * CHUNK_BYTES;    // two stages
  static constexpr int NSTG = 3;                                // dQ staging buffers in flight
  static constexpr int STG_OFF = AUX_OFF + 2 * AUX_BYTES;      // dQ staging: NSTG x [4][128][4] fp32
  static constexpr int STG_BYTES = 16 * TILE * 4;
  static constexpr int LIST_OFF = STG_OFF + NSTG * STG_BYTES;  // int32 query tiles of the column
  static constexpr int LCLS_OFF = LIST_OFF + kMaxList * 4;     // uint8 their tile classes
  static constexpr int BAR_OFF = LCLS_OFF + kMaxList;
  static constexpr int NBAR = 21;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;
  static_assert(SMEM_ALLOC <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
  // split columns: a CTA of rank > 0 leaves its fp32 dV, dK partial here after its main loop
  // ([2][TILE][PART_ROW], rows padded by 16 bytes), over the K / V / Q / dO buffers, which are
  // free by then; the dQ staging ring (still draining) lies beyond it
  static constexpr int PART_ROW = HD + 4;
  static constexpr int PART_OFF = 0;
  static constexpr int PART_BYTES = 2 * TILE * PART_ROW * 4;
  static_assert(PART_OFF + PART_BYTES <= STG_OFF, "partial-sum area must not overlap the dQ staging ring");
  // 16 warps = 4 warpgroups: [producer, MMA, 2 idle] [4 dQ drain] [4 + 4 elementwise]
  static constexpr int THREADS = 512;
  static constexpr int LAUNCH_REGS = 128;                      // 512 x 128 = the whole register file
  static constexpr int REGS_CTRL = 88, REGS_DRAIN = 160, REGS_EW = 128;
  static_assert(128 * REGS_CTRL + 128 * REGS_DRAIN + 256 * REGS_EW <= THREADS * LAUNCH_REGS,
                "register re-balancing must fit the launch allocation");
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns: S^T in A (P^T packed bf16 over it, query half g at 64 g), dP^T and dQ in B
  static constexpr uint32_t A_COL = 0, B_COL = 128, DV_COL = 256, DK_COL = 256 + HD;
  static constexpr uint32_t IDESC_SDP = idesc_bf16(TILE, TILE, 0, 0);   // K/V K-major, Q/dO K-major
  static constexpr uint32_t IDESC_DKV = idesc_bf16(TILE, HD, 0, 1);     // P^T (TMEM) / dS^T K-major, dO/Q MN-major
  static constexpr uint32_t IDESC_DQ = idesc_bf16(TILE, HD, 1, 1);      // dS MN-major, K MN-major
  static constexpr uint32_t KV_TX = 2 * NCH * CHUNK_BYTES;
  static constexpr uint32_t Q_TX = NCH * CHUNK_BYTES;
  static constexpr uint32_t DO_TX = NCH * CHUNK_BYTES;
};

struct BwdParams {
  const int32_t* col_ptr;
  const int32_t* col_idx;
  const int32_t* col_order;
  const int32_t* tok_in;
  const int32_t* tok_out;
  const int32_t* pos;
  const int32_t* tile_runs;
  const int32_t* tile_nruns;
  const uint8_t* tile_class;
  const float* nlse2;        // [Hq][Npad] -LSE log2e
  const float* ndlt;         // [Hq][Npad] -delta scale
  float* dqacc;              // [Hq][T][HD/4][128][4]: one contiguous 64 KiB block per (head, query tile)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t* status;
  int N, T, Npad, Hq, Hkv, grp;
  float scale, scale_log2, rope_theta;
  int gw_len, gw_tiles;      // gateway prefix (0 = none): its key tiles get CTAs of their own
  int split;                 // CTAs per column (a cluster): CTA s takes steps s, s + split, ...
  float* dk_gw;              // [gw_len][Hkv][HD] fp32, accumulated (+=); rotated back at pos = row
  float* dv_gw;
  uint64_t wait_ns;
};

DEVI uint8_t* align1024b(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

DEVI void mbar_wait_drain_b(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return;
}

// ------------------------------------------------------------------------------------------
// per query row: -delta scale (delta_i = sum_c dO_ic O_ic) and -LSE log2e, and zeroes of the
// same rows of the dQ accumulator.  With per-token weights w the input is U, dO = w U: delta is
// then sum_c U_ic O_ic and log2 w_i is added to the -LSE log2e term, which folds the weight into
// P (P w, exact up to rounding), so that dS = (P w)(dP(U) - delta(U)) and dV = sum (P w)^T U are
// the gradients for dO without dO being formed.  One block per (32 tokens, q head): 8 threads per token
// each dot 16 columns (two 16-byte loads of O and of dO, a 256-byte row per token), so the
// per-head outputs are written as coalesced 128-byte rows.
template <int HD>
__global__ void __launch_bounds__(256) k_bwd_pre(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                                                 const float* __restrict__ lse, const float* __restrict__ w,
                                                 float* ndlt, float* nlse2, float scale, float* dqacc, int N, int Npad,
                                                 int Hq) {
  constexpr int TPT = 8, VPT = HD / 8 / TPT;      // threads per token, 16-byte vectors per thread
  const int h = blockIdx.y;
  const int tok = blockIdx.x * 32 + threadIdx.x / TPT;
  const int sub = threadIdx.x % TPT;
  float acc = 0.f;
  if (tok < N) {
    const size_t base = ((size_t)tok * Hq + h) * (HD / 8) + sub * VPT;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const uint4 a = o[base + v], b = dO[base + v];
      acc += bf16lo(a.x) * bf16lo(b.x) + bf16hi(a.x) * bf16hi(b.x) + bf16lo(a.y) * bf16lo(b.y) +
             bf16hi(a.y) * bf16hi(b.y) + bf16lo(a.z) * bf16lo(b.z) + bf16hi(a.z) * bf16hi(b.z) +
             bf16lo(a.w) * bf16lo(b.w) + bf16hi(a.w) * bf16hi(b.w);
    }
  }
#pragma unroll
  for (int off = TPT / 2; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (sub == 0 && tok < Npad) {
    const size_t at = (size_t)h * Npad + tok;
    ndlt[at] = tok < N ? -acc * scale : 0.f;
    // with per-token weights (dO = w U, U given): P w = 2^(S scale log2e - LSE log2e + log2 w)
    nlse2[at] = -lse[at] * 1.4426950408889634f + ((w && tok < N) ? log2f(w[tok]) : 0.f);
  }
  // dQ accumulator rows of these 32 tokens for head h: [HD/4][128][4] block of (h, query tile),
  // 32 consecutive rows = 512 contiguous bytes per 4 columns
  const int t0 = blockIdx.x * 32;
  float4* blk = reinterpret_cast<float4*>(dqacc + ((size_t)h * (Npad / TILE) + t0 / TILE) * HD * TILE) + (t0 % TILE);
  for (int e = threadIdx.x; e < (HD / 4) * 32; e += blockDim.x)
    blk[(size_t)(e / 32) * TILE + (e % 32)] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(BwdCfg<HD>::THREADS, 1)
    k_bwd_dkdv(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmKg, const __grid_constant__ CUtensorMap tmVg,
               const BwdParams p) {
  using C = BwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024b(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* kv_full = bars + 0;
  uint64_t* do_full = bars + 1;
  uint64_t* do_empty = bars + 2;
  uint64_t* s_full = bars + 3;                  // S^T(n) in A
  uint64_t* dp_full = bars + 4;                 // dP^T(n) in B
  uint64_t* dq_full = bars + 5;
  uint64_t* dq_free = bars + 6;
  uint64_t* dkdv_done = bars + 7;
  uint64_t* drain = bars + 8;
  uint64_t* aux_full = bars + 9;                // [2] row data of a step (LSE, delta, dfs_in, runs)
  uint64_t* aux_empty = bars + 11;              // [2] one arrival per elementwise warp after dS
  uint64_t* p_ready = bars + 13;                // P^T of both groups written
  uint64_t* ds_ready = bars + 14;               // dS^T of both groups written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  int* abort_flag = reinterpret_cast<int*>(sm + C::MISC_OFF + 4);
  int32_t* list_s = reinterpret_cast<int32_t*>(sm + C::LIST_OFF);
  uint8_t* lcls_s = sm + C::LCLS_OFF;

  uint64_t* peer_ready = bars + 15;            // rank 0: the other ranks' partials are in place
  uint64_t* peer_done = bars + 16;             // rank > 0: rank 0 has read this CTA's partial
  uint64_t* qs_full = bars + 17;               // Q for S^T(n) landed
  uint64_t* qs_empty = bars + 18;              // S^T(n) done: that buffer is free
  uint64_t* qd_full = bars + 19;               // Q for dK(n) landed
  uint64_t* qd_empty = bars + 20;              // dK(n) done: that buffer is free
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // clusters of p.split CTAs share one column: rank s takes its steps s, s + split, ...
  const int srank = p.split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int u = blockIdx.x / p.split;
  // CTAs [0, gw_tiles Hkv): gateway key tiles, seen by every query tile of the partition
  // (they also have the longest columns, so they start first); then the own key tiles.
  const int ngw = p.gw_tiles * p.Hkv;
  const bool gwc = u < ngw;
  const int kt = gwc ? u / p.Hkv : p.col_order[(u - ngw) / p.Hkv];
  const int kvh = u % p.Hkv;
  const int cp0 = gwc ? 0 : p.col_ptr[kt];
  const int ccnt = gwc ? p.T : p.col_ptr[kt + 1] - cp0;
  const int gw_cls = (gwc && kt == p.gw_tiles - 1 && (p.gw_len % TILE) != 0) ? 1 : 2;
  const int total_all = ccnt * p.grp;           // steps: query tile (outer, descending) x q head (inner)
  const int eff = p.split;                      // CTAs the column's steps are dealt to
  const int total = total_all > srank ? (total_all - srank + eff - 1) / eff : 0;   // this CTA's steps

  // the column's query tiles and their classes, staged once
  for (int i = threadIdx.x; i < ccnt && i < kMaxList; i += blockDim.x) {
    const int qt = gwc ? i : p.col_idx[cp0 + i];
    list_s[i] = qt;
    // class in bits 0-1, the query tile's node-run count (capped at TREE_MAX_RUNS + 1) in bits 3-7,
    // so the mask of a partial step reads no global memory
    lcls_s[i] = gwc ? gw_cls
                    : static_cast<uint8_t>(p.tile_class[(size_t)qt * p.T + kt] |
                                           (min(p.tile_nruns[qt], TREE_MAX_RUNS + 1) << 3));
  }
  // step n -> (q head, query tile, class).  Query tiles are walked from the end of the column
  // with the group's q heads innermost, so CTAs running at the same time (whatever their key
  // tile) reach the same (query tile, head) pairs together and their dQ lines stay in L2.
  auto step_tile = [&](int n, int& h, int& qt, int& cls) {
    const int gn = srank + n * eff;             // the step's index in the whole column
    const int i = ccnt - 1 - gn / p.grp;
    h = kvh * p.grp + gn % p.grp;
    if (i < kMaxList) { qt = list_s[i]; cls = lcls_s[i] & 7; }
    else if (gwc) { qt = i; cls = gw_cls; }
    else { qt = p.col_idx[cp0 + i]; cls = p.tile_class[(size_t)qt * p.T + kt]; }
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&aux_full[i], 1); mbar_init(&aux_empty[i], 8); }
    mbar_init(qs_full, 1);
    mbar_init(qs_empty, 1);
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 8);                      // one arrival per elementwise warp
    mbar_init(ds_ready, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);                      // one arrival per drain warp
    mbar_init(dkdv_done, 1);
    mbar_init(drain, 1);
    mbar_init(peer_ready, eff > 1 ? eff - 1 : 1);
    mbar_init(peer_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (p.split > 1) {
    __syncthreads();
    cluster_sync_all();                         // every CTA's barriers initialised before remote arrivals
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

  if (warp < 4) {
    regs_dec<C::REGS_CTRL>();
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmDO);
      mbar_expect_tx(kv_full, C::KV_TX);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(sm + C::K_OFF + c * CHUNK_BYTES, gwc ? &tmKg : &tmK, kv_full, c * 64, kvh, kt * TILE);
        tma_load_3d(sm + C::V_OFF + c * CHUNK_BYTES, gwc ? &tmVg : &tmV, kv_full, c * 64, kvh, kt * TILE);
      }
      // Q tile of step m into the buffer of the S product (which = 0) or of the dK product (1)
      auto load_q = [&](int m, int which) {
        int h, qt, cls;
        step_tile(m, h, qt, cls);
        uint64_t* bar = which ? qd_full : qs_full;
        mbar_expect_tx(bar, C::Q_TX);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sm + C::Q_OFF + (which * C::NCH + c) * CHUNK_BYTES, &tmQ, bar, c * 64, h, qt * TILE);
      };
      auto load_aux = [&](int m) {             // row data of step m into ring stage m % 2
        int h, qt, cls;
        step_tile(m, h, qt, cls);
        uint64_t* bar = &aux_full[m & 1];
        mbar_expect_tx(bar, C::AUX_BYTES);
        uint8_t* aux = sm + C::AUX_OFF + (m & 1) * C::AUX_BYTES;
        const size_t lo = (size_t)h * p.Npad + (size_t)qt * TILE;
        bulk_load(aux + C::AUX_LSE, p.nlse2 + lo, TILE * 4, bar);
        bulk_load(aux + C::AUX_DLT, p.ndlt + lo, TILE * 4, bar);
        bulk_load(aux + C::AUX_QIN, p.tok_in + (size_t)qt * TILE, TILE * 4, bar);
        bulk_load(aux + C::AUX_RUNS, p.tile_runs + (size_t)qt * TREE_MAX_RUNS * 4, TREE_MAX_RUNS * 16, bar);
      };
      // Loads in the order their buffers free up during step n: dO(n) after dV(n-1), Q for
      // S(n+1) after S(n), the row data of step n+1 after step n-1's dS, Q for dK(n) after dK(n-1).
      int qs_issued = 0, qd_issued = 0, aux_issued = 0, do_issued = 0;
      if (total > 0) {
        load_q(0, 0);
        load_aux(0);
        load_q(0, 1);
        qs_issued = qd_issued = aux_issued = 1;
      }
      if (total > 1) { load_aux(1); aux_issued = 2; }
      for (int n = 0; n < total; ++n) {
        int h, qt, cls;
        step_tile(n, h, qt, cls);
        // dO of step n once dV(n-1) and dP(n-1) have read the buffer
        if (n > 0 && !mbar_wait(do_empty, (n - 1) & 1, wc)) break;
        mbar_expect_tx(do_full, C::DO_TX);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sm + C::DO_OFF + c * CHUNK_BYTES, &tmDO, do_full, c * 64, h, qt * TILE);
        do_issued = n + 1;
        if (n + 1 < total) {
          if (!mbar_wait(qs_empty, n & 1, wc)) break;
          load_q(n + 1, 0);
          qs_issued = n + 2;
          // stage (n+1) % 2 held step n-1's row data until its dS phase ended
          if (n >= 1) {
            if (!mbar_wait(&aux_empty[(n + 1) & 1], ((n - 1) >> 1) & 1, wc)) break;
            load_aux(n + 1);
            aux_issued = n + 2;
          }
        }
        if (n > 0) {
          if (!mbar_wait(qd_empty, (n - 1) & 1, wc)) break;
          load_q(n, 1);
          qd_issued = n + 1;
        }
      }
      if (*abort_flag) {
        mbar_wait_drain_b(kv_full, 0, p.wait_ns);
        if (do_issued > 0) mbar_wait_drain_b(do_full, (do_issued - 1) & 1, p.wait_ns);
        if (qs_issued > 0) mbar_wait_drain_b(qs_full, (qs_issued - 1) & 1, p.wait_ns);
        if (qd_issued > 0) mbar_wait_drain_b(qd_full, (qd_issued - 1) & 1, p.wait_ns);
        for (int m = (aux_issued > 2 ? aux_issued - 2 : 0); m < aux_issued; ++m)
          mbar_wait_drain_b(&aux_full[m & 1], (m >> 1) & 1, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // operand descriptors, built once: K-major (LBO unused) and MN-major (LBO = 64-element block)
      const uint32_t k_base = smem_u32(sm + C::K_OFF), v_base = smem_u32(sm + C::V_OFF);
      const uint32_t do_base = smem_u32(sm + C::DO_OFF), dst_base = smem_u32(sm + C::DST_OFF);
      const uint32_t q_base0 = smem_u32(sm + C::Q_OFF), q_base1 = q_base0 + C::NCH * CHUNK_BYTES;
      const uint64_t k_km = sdesc_sw128(k_base, 16, 1024), k_mn = sdesc_sw128(k_base, CHUNK_BYTES, 1024);
      const uint64_t v_km = sdesc_sw128(v_base, 16, 1024);
      const uint64_t do_km = sdesc_sw128(do_base, 16, 1024), do_mn = sdesc_sw128(do_base, CHUNK_BYTES, 1024);
      const uint64_t ds_km = sdesc_sw128(dst_base, 16, 1024), ds_mn = sdesc_sw128(dst_base, CHUNK_BYTES, 1024);
      const uint64_t qs_km = sdesc_sw128(q_base0, 16, 1024);             // Q for S, K-major
      const uint64_t qd_mn = sdesc_sw128(q_base1, CHUNK_BYTES, 1024);    // Q for dK, MN-major
      // Software-pipelined over the steps so the tensor core runs one step's GEMMs while the
      // elementwise warps work on the other step's tile.  A holds S^T(n), then P^T(n) until dV(n);
      // B holds dP^T(n) until dS(n) is computed, then dQ(n) until the drain has read it.  Issue
      // order for step n: [dQ(n-1), dK(n-1)], dP(n), dV(n), S(n+1).
      auto issue_s = [&](int m) -> bool {       // S^T(m) = K Q(m)^T into A
        if (!mbar_wait(qs_full, m & 1, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
          umma_bf16(tmem + C::A_COL, sdesc_adv(k_km, off), sdesc_adv(qs_km, off), C::IDESC_SDP, kk > 0 ? 1u : 0u);
        }
        umma_commit(s_full);
        umma_commit(qs_empty);                                   // Q for S free for step m+1
        return true;
      };
      // dQ(m) = dS(m) K into B first, so the drain copies it out while dK += dS(m)^T Q(m) runs
      auto issue_dq_dk = [&](int m) -> bool {
        if (!mbar_wait(ds_ready, m & 1, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          umma_bf16(tmem + C::B_COL, sdesc_adv(ds_mn, kk * 16 * 128), sdesc_adv(k_mn, kk * 16 * 128), C::IDESC_DQ,
                    kk > 0 ? 1u : 0u);
        umma_commit(dq_full);
        if (!mbar_wait(qd_full, m & 1, wc)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          umma_bf16(tmem + C::DK_COL, sdesc_adv(ds_km, (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32),
                    sdesc_adv(qd_mn, kk * 16 * 128), C::IDESC_DKV, (m > 0 || kk > 0) ? 1u : 0u);
        umma_commit(qd_empty);                                   // Q for dK free for step m+1
        return true;
      };
      bool ok = mbar_wait(kv_full, 0, wc);
      if (ok && total > 0) ok = issue_s(0);
      for (int n = 0; ok && n < total; ++n) {
        if (n > 0 && !issue_dq_dk(n - 1)) { ok = false; break; }
        // dP^T(n) = V dO(n)^T into B once the drain has read dQ(n-1): it runs while the
        // elementwise warps compute P(n), so dS(n) can follow P(n) without a gap
        if (!mbar_wait(do_full, n & 1, wc)) { ok = false; break; }
        if (n > 0 && !mbar_wait(dq_free, (n - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;
          umma_bf16(tmem + C::B_COL, sdesc_adv(v_km, off), sdesc_adv(do_km, off), C::IDESC_SDP, kk > 0 ? 1u : 0u);
        }
        umma_commit(dp_full);
        // dV += P(n)^T dO(n), P^T read from TMEM
        if (!mbar_wait(p_ready, n & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          umma_bf16_tmem_a(tmem + C::DV_COL, tmem + C::A_COL + (kk >> 2) * 64 + (kk & 3) * 8,
                           sdesc_adv(do_mn, kk * 16 * 128), C::IDESC_DKV, (n > 0 || kk > 0) ? 1u : 0u);
        umma_commit(do_empty);                                   // dO(n) free once dP(n), dV(n) are done
        if (n + 1 < total && !issue_s(n + 1)) { ok = false; break; }
      }
      if (ok && total > 0) ok = issue_dq_dk(total - 1);
      if (ok) umma_commit(dkdv_done);
      umma_commit(drain);
      mbar_wait_drain_b(drain, 0, p.wait_ns);
    }
  }
  } else if (warp < 8) {
    regs_inc<C::REGS_DRAIN>();
    // ---------------------------------------------------------------- dQ drain warpgroup
    // Thread r copies dQ(n) row r (all HD columns) out of TMEM and frees the columns for
    // dP(n+1).  The rows then go to the fp32 accumulator 16 columns (8 KiB) at a time through a
    // three-buffer shared staging ring and a bulk reduce-add by the TMA unit, while the next
    // step runs: no per-element atomics compete with the tensor-core issue for the memory pipe.
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float* stg = reinterpret_cast<float*>(sm + C::STG_OFF);
    const bool leader = (threadIdx.x == 128);
    int groups = 0;                               // bulk groups committed by the leader
    int stage_slot = 0;                           // next staging buffer (same on every drain thread)
    for (int n = 0; n < total; ++n) {
      int h, qt, cls;
      step_tile(n, h, qt, cls);
      // all four warps agree before the named barriers below, so a timeout cannot split them
      if (!named_bar_and(1, 128, mbar_wait_warp(dq_full, n & 1, wc))) break;
      tc_fence_after();
      uint32_t qv[HD];
#pragma unroll
      for (int jc = 0; jc < HD / 32; ++jc)
        tmem_ld32(tmem + lane_off + C::B_COL + 32 * jc, *reinterpret_cast<uint32_t(*)[32]>(qv + 32 * jc));
#pragma unroll
      for (int jc = 0; jc < HD / 32; ++jc) tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(qv + 32 * jc));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      // [HD/4][128][4] block of (h, qt); rows past the last token carry exact zeros
      float* blk = p.dqacc + ((size_t)h * p.T + qt) * HD * TILE;
#pragma unroll
      for (int gi = 0; gi < HD / 16; ++gi) {
        // staging buffer of the drain's running group count: the reduce that last read it is
        // the third-newest, so two reduces stay queued for the TMA unit while this one is filled
        const int slot = stage_slot;
        stage_slot = (stage_slot + 1 == C::NSTG) ? 0 : stage_slot + 1;
        float* buf = stg + slot * (C::STG_BYTES / 4);
        if (leader && groups >= C::NSTG) bulk_wait_group_read2();
        named_bar_sync(1, 128);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(buf + (j * TILE + r) * 4) =
              make_uint4(qv[16 * gi + 4 * j], qv[16 * gi + 4 * j + 1], qv[16 * gi + 4 * j + 2], qv[16 * gi + 4 * j + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          bulk_reduce_add_f32(blk + (size_t)gi * 4 * TILE * 4, buf, C::STG_BYTES);
          bulk_commit_group();
          ++groups;
        }
      }
    }
    if (leader) bulk_wait_group0();               // every reduce has landed before the CTA ends
  } else {
    regs_inc<C::REGS_EW>();
    // ---------------------------------------------------------------- elementwise warps
    // Two warpgroups share the 128 TMEM lanes: group g takes query columns [64 g, 64 g + 64)
    // of S^T / dP^T, and output columns [HD/2 g, HD/2 (g+1)) of dV, pairs of dK.
    const int g = (warp - 8) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;                 // key row (S^T, dP^T, dK, dV) or query row (dQ)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int j = kt * TILE + r;                  // key token (a gateway row in a gateway CTA)
    const int kin = gwc ? 0 : p.tok_in[j], kout = gwc ? 0 : p.tok_out[j];
    const uint64_t nl2e2 = f2_pack(-1.4426950408889634f, -1.4426950408889634f);
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t sc2 = f2_pack(p.scale, p.scale), nsc2 = f2_pack(-p.scale, -p.scale);
    bool ok = true;
    for (int n = 0; n < total; ++n) {
      int h, qt, cls;
      step_tile(n, h, qt, cls);
      if (!mbar_wait_warp(&aux_full[n & 1], (n >> 1) & 1, wc) || !mbar_wait_warp(s_full, n & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const uint8_t* aux = sm + C::AUX_OFF + (n & 1) * C::AUX_BYTES;
      const float* nlse_s = reinterpret_cast<const float*>(aux + C::AUX_LSE);
      const float* ndlt_s = reinterpret_cast<const float*>(aux + C::AUX_DLT);
      const int jrel = j - qt * TILE;             // query i is causal-visible iff i >= jrel
      // partial tile: bits of this group's 64 query columns that key j may see, one
      // ancestor-interval test per node run of the query tile
      uint32_t vw0 = 0xffffffffu, vw1 = 0xffffffffu;
      if (cls == 1 && gwc) {                      // ragged gateway tile: keys past gw_len see nothing
        vw0 = vw1 = (j < p.gw_len) ? 0xffffffffu : 0u;
      } else if (cls == 1) {
        uint32_t vm[4] = {0u, 0u, 0u, 0u};
        const int gi = ccnt - 1 - (srank + n * eff) / p.grp;   // the step's place in the column
        const int nr = gi < kMaxList ? static_cast<int>(lcls_s[gi] >> 3) : p.tile_nruns[qt];
        if (nr <= TREE_MAX_RUNS) {
          const int4* runs = reinterpret_cast<const int4*>(aux + C::AUX_RUNS);
          for (int k = 0; k < nr; ++k) {
            const int4 rn = runs[k];
            if (kin <= rn.z && rn.z <= kout) set_bits(vm, rn.x, rn.y);
          }
        } else {
          const int32_t* qin_s = reinterpret_cast<const int32_t*>(aux + C::AUX_QIN);
          for (int c4 = 0; c4 < TILE / 4; ++c4) {
            const int4 q4 = *reinterpret_cast<const int4*>(qin_s + 4 * c4);
            const uint32_t bits = (uint32_t)(kin <= q4.x && q4.x <= kout) | ((uint32_t)(kin <= q4.y && q4.y <= kout) << 1) |
                                  ((uint32_t)(kin <= q4.z && q4.z <= kout) << 2) |
                                  ((uint32_t)(kin <= q4.w && q4.w <= kout) << 3);
            vm[c4 >> 3] |= bits << (4 * (c4 & 7));
          }
        }
        set_bits_clear_below(vm, jrel);
        vw0 = g ? vm[2] : vm[0];
        vw1 = g ? vm[3] : vm[1];
      }
      // P phase: P = exp2(S scale log2e - LSE log2e) for this group's 64 query columns: all
      // four S^T loads in flight at once, P^T back into A as packed bf16 for dV, P kept in
      // registers in fp32 for dS.
      float pf[64];
      {
        uint32_t sv[64];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tmem_ld16(tmem + lane_off + C::A_COL + 64 * g + 16 * k, *reinterpret_cast<uint32_t(*)[16]>(sv + 16 * k));
#pragma unroll
        for (int k = 0; k < 4; ++k) tmem_wait_ld16(*reinterpret_cast<uint32_t(*)[16]>(sv + 16 * k));
        if (cls == 1) {                           // invisible pairs: S = -inf, so P = 2^-inf = 0
          const uint32_t vw[2] = {vw0, vw1};
          apply_mask_words<2>(sv, vw, __float_as_uint(-INFINITY));
        }
        uint32_t pp[32];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nlse_s + 64 * g + c);
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, f2_pack(l4.x, l4.y)), x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2x2, f2_pack(l4.z, l4.w)), x2, x3);
          float pv[4] = {ex2_approx(x0), ex2_approx(x1), ex2_approx(x2), ex2_approx(x3)};
#pragma unroll
          for (int e = 0; e < 4; ++e) pf[c + e] = pv[e];
          pp[c >> 1] = pack_bf16(pv[0], pv[1]);
          pp[(c >> 1) + 1] = pack_bf16(pv[2], pv[3]);
        }
        // P^T: 32 packed columns over this group's (already read) S^T columns
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tmem_store8(tmem + lane_off + C::A_COL + 64 * g + 8 * k, *reinterpret_cast<const uint32_t(*)[8]>(pp + 8 * k));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);
      }
      // dS phase: dS = P (dP scale - delta scale), written as bf16 dS^T (keys x queries) for dK
      // and dQ
      if (!mbar_wait_warp(dp_full, n & 1, wc)) { ok = false; break; }
      tc_fence_after();
      {
        uint8_t* dsb = sm + C::DST_OFF + g * CHUNK_BYTES;
#pragma unroll
        for (int half = 0; half < 2; ++half) {    // 32 query columns at a time (register budget)
          uint32_t dv[32];
          tmem_ld16(tmem + lane_off + C::B_COL + 64 * g + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(dv));
          tmem_ld16(tmem + lane_off + C::B_COL + 64 * g + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(dv + 16));
          tmem_wait_ld16x2(*reinterpret_cast<uint32_t(*)[16]>(dv), *reinterpret_cast<uint32_t(*)[16]>(dv + 16));
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int k = 2 * half + k2;
            uint32_t dd[8];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
              const int cc = 16 * k + c, cl = 16 * k2 + c;
              const float4 d4 = *reinterpret_cast<const float4*>(ndlt_s + 64 * g + cc);
              const uint64_t t01 = f2_fma(f2_pack(__uint_as_float(dv[cl]), __uint_as_float(dv[cl + 1])), sc2, f2_pack(d4.x, d4.y));
              const uint64_t t23 = f2_fma(f2_pack(__uint_as_float(dv[cl + 2]), __uint_as_float(dv[cl + 3])), sc2, f2_pack(d4.z, d4.w));
              float e0, e1, e2, e3;
              f2_unpack(f2_mul(f2_pack(pf[cc], pf[cc + 1]), t01), e0, e1);
              f2_unpack(f2_mul(f2_pack(pf[cc + 2], pf[cc + 3]), t23), e2, e3);
              dd[c >> 1] = pack_bf16(e0, e1);
              dd[(c >> 1) + 1] = pack_bf16(e2, e3);
            }
            st_swizzled_unit(dsb, r, 2 * k, make_uint4(dd[0], dd[1], dd[2], dd[3]));
            st_swizzled_unit(dsb, r, 2 * k + 1, make_uint4(dd[4], dd[5], dd[6], dd[7]));
          }
        }
        tc_fence_before();                        // the dP^T reads are done before dQ rewrites B
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(ds_ready);
          mbar_arrive(&aux_empty[n & 1]);         // this step's row data no longer read
        }
      }
    }
    // -------------------------------------------------------------- epilogue: dV, dK rows
    // With split columns the cluster's ranks > 0 leave their fp32 partials in shared memory and
    // rank 0 adds them, in rank order, to its own before the write-out: the same sum whatever
    // the timing, and nothing accumulated in global memory.
    const bool have = ok && mbar_wait_warp(dkdv_done, 0, wc);
    if (have) tc_fence_after();
    const uint32_t part_s = smem_u32(sm + C::PART_OFF);
    auto part_at = [&](int which, int col) -> uint32_t {   // which: 0 dV, 1 dK; this thread's row r
      return part_s + static_cast<uint32_t>(((which * TILE + r) * C::PART_ROW + col) * 4);
    };
    if (eff > 1 && srank > 0) {
      if (have) {
        // a rank with no steps of the column (a short column) never wrote its accumulators:
        // its partial is zero
        const uint32_t keep = total > 0 ? 0xffffffffu : 0u;
#pragma unroll 1
        for (int jc = 0; jc < HD / 64; ++jc) {
          const int c0 = (HD / 2) * g + 32 * jc;
          uint32_t a[32];
          tmem_load32(tmem + lane_off + C::DV_COL + c0, a);
#pragma unroll
          for (int c = 0; c < 32; ++c) a[c] &= keep;
#pragma unroll
          for (int v = 0; v < 8; ++v) st_shared_v4(part_at(0, c0 + 4 * v), a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
        }
#pragma unroll 1
        for (int jc = 0; jc < HD / 64; ++jc) {
          const int c0 = (HD / 4) * g + 16 * jc;
          uint32_t a[16], b[16];
          tmem_load16(tmem + lane_off + C::DK_COL + c0, a);
          tmem_load16(tmem + lane_off + C::DK_COL + HD / 2 + c0, b);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            a[c] &= keep;
            b[c] &= keep;
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            st_shared_v4(part_at(1, c0 + 4 * v), a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
            st_shared_v4(part_at(1, HD / 2 + c0 + 4 * v), b[4 * v], b[4 * v + 1], b[4 * v + 2], b[4 * v + 3]);
          }
        }
      }
      named_bar_sync(2, 256);                     // every elementwise thread's rows are in place
      if (threadIdx.x == 256) mbar_arrive_remote(mapa_shared(smem_u32(peer_ready), 0));
      (void)mbar_wait_cluster(peer_done, 0, wc);  // rank 0 reads this area until it arrives here
    } else {
      int nsum = 1;                               // ranks summed: this one, then 1 .. eff-1
      if (eff > 1) nsum = __all_sync(0xffffffffu, mbar_wait_cluster(peer_ready, 0, wc)) ? eff : 1;
      if (have && gwc) {
        // gateway row j: dV and (rotated back at position j, the row's index on the path from
        // the root) dK added in fp32 to the caller's accumulators, which sum over child partitions
        const bool live = j < p.gw_len;
        float* dvg = p.dv_gw + ((size_t)j * p.Hkv + kvh) * HD;
#pragma unroll 1
        for (int jc = 0; jc < HD / 64; ++jc) {
          const int c0 = (HD / 2) * g + 32 * jc;
          uint32_t a[32];
          tmem_load32(tmem + lane_off + C::DV_COL + c0, a);
          float f[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) f[c] = __uint_as_float(a[c]);
          add_cluster_partials(f, part_at(0, c0), nsum);
          if (live) {
            float4* d4 = reinterpret_cast<float4*>(dvg + c0);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              float4 t = d4[v];
              t.x += f[4 * v];
              t.y += f[4 * v + 1];
              t.z += f[4 * v + 2];
              t.w += f[4 * v + 3];
              d4[v] = t;
            }
          }
        }
        float* dkg = p.dk_gw + ((size_t)j * p.Hkv + kvh) * HD;
        const float posf = static_cast<float>(j);
#pragma unroll 1
        for (int jc = 0; jc < HD / 64; ++jc) {
          const int c0 = (HD / 4) * g + 16 * jc;
          uint32_t a[16], b[16];
          tmem_load16(tmem + lane_off + C::DK_COL + c0, a);
          tmem_load16(tmem + lane_off + C::DK_COL + HD / 2 + c0, b);
          float lo[16], hi[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            lo[c] = __uint_as_float(a[c]);
            hi[c] = __uint_as_float(b[c]);
          }
          add_cluster_partials(lo, part_at(1, c0), nsum);
          add_cluster_partials(hi, part_at(1, HD / 2 + c0), nsum);
          if (live) {
            if (p.rope_theta > 0.f) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                float sv, cv;
                sincosf(posf * rope_inv_freq(c0 + c, HD, p.rope_theta), &sv, &cv);
                const float g1 = lo[c], g2 = hi[c];
                lo[c] = g1 * cv + g2 * sv;
                hi[c] = g2 * cv - g1 * sv;
              }
            }
            // 16 consecutive fp32 of each half row: four 16-byte read-add-writes per half
            float4* d4 = reinterpret_cast<float4*>(dkg + c0);
            float4* e4 = reinterpret_cast<float4*>(dkg + HD / 2 + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float4 t = d4[v], w = e4[v];
              t.x += lo[4 * v]; t.y += lo[4 * v + 1]; t.z += lo[4 * v + 2]; t.w += lo[4 * v + 3];
              w.x += hi[4 * v]; w.y += hi[4 * v + 1]; w.z += hi[4 * v + 2]; w.w += hi[4 * v + 3];
              d4[v] = t;
              e4[v] = w;
            }
          }
        }
      }
      if (have && !gwc) {
        // dV row j, columns [HD/2 g, HD/2 (g+1))
        __nv_bfloat16* dvrow = p.dv + ((size_t)j * p.Hkv + kvh) * HD;
#pragma unroll 1
        for (int jc = 0; jc < HD / 64; ++jc) {
          const int c0 = (HD / 2) * g + 32 * jc;
          uint32_t a[32];
          tmem_load32(tmem + lane_off + C::DV_COL + c0, a);
          float f[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) f[c] = __uint_as_float(a[c]);
          add_cluster_partials(f, part_at(0, c0), nsum);
          if (j < p.N) {
            uint4* d4 = reinterpret_cast<uint4*>(dvrow + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              d4[v] = make_uint4(pack_bf16(f[8 * v + 0], f[8 * v + 1]), pack_bf16(f[8 * v + 2], f[8 * v + 3]),
                                 pack_bf16(f[8 * v + 4], f[8 * v + 5]), pack_bf16(f[8 * v + 6], f[8 * v + 7]));
          }
        }
        // dK row j with the inverse RoPE rotation: group g takes the pairs (c, c + HD/2),
        // c in [HD/4 g, HD/4 (g+1))
        __nv_bfloat16* dkrow = p.dk + ((size_t)j * p.Hkv + kvh) * HD;
        const float posf = (j < p.N) ? static_cast<float>(p.pos[j]) : 0.f;
#pragma unroll 1
        for (int jc = 0; jc < HD / 64; ++jc) {
          const int c0 = (HD / 4) * g + 16 * jc;
          uint32_t a[16], b[16];
          tmem_load16(tmem + lane_off + C::DK_COL + c0, a);
          tmem_load16(tmem + lane_off + C::DK_COL + HD / 2 + c0, b);
          float lo[16], hi[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            lo[c] = __uint_as_float(a[c]);
            hi[c] = __uint_as_float(b[c]);
          }
          add_cluster_partials(lo, part_at(1, c0), nsum);
          add_cluster_partials(hi, part_at(1, HD / 2 + c0), nsum);
          if (p.rope_theta > 0.f) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float sv, cv;
              sincosf(posf * rope_inv_freq(c0 + c, HD, p.rope_theta), &sv, &cv);
              const float g1 = lo[c], g2 = hi[c];
              lo[c] = g1 * cv + g2 * sv;
              hi[c] = g2 * cv - g1 * sv;
            }
          }
          if (j < p.N) {
            uint4* d4 = reinterpret_cast<uint4*>(dkrow + c0);
            uint4* e4 = reinterpret_cast<uint4*>(dkrow + HD / 2 + c0);
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              d4[v] = make_uint4(pack_bf16(lo[8 * v], lo[8 * v + 1]), pack_bf16(lo[8 * v + 2], lo[8 * v + 3]),
                                 pack_bf16(lo[8 * v + 4], lo[8 * v + 5]), pack_bf16(lo[8 * v + 6], lo[8 * v + 7]));
              e4[v] = make_uint4(pack_bf16(hi[8 * v], hi[8 * v + 1]), pack_bf16(hi[8 * v + 2], hi[8 * v + 3]),
                                 pack_bf16(hi[8 * v + 4], hi[8 * v + 5]), pack_bf16(hi[8 * v + 6], hi[8 * v + 7]));
            }
          }
        }
      }
      if (eff > 1) {
        named_bar_sync(2, 256);                   // every thread has read the other ranks' areas
        if (threadIdx.x == 256)
          for (int q = 1; q < eff; ++q) mbar_arrive_remote(mapa_shared(smem_u32(peer_done), q));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------
// dQ = R(pos)^T dQacc: one block per (32 tokens, group of up to 8 q heads); angles computed
// once per token and block.
// Per head: the 32 rows of the [d/4][128][4] block are read with 16-byte loads (4 columns of
// one row each; 32 threads cover 512 contiguous bytes), transposed through shared memory,
// rotated, and written as 16-byte bf16 stores.
template <int HD>
__global__ void __launch_bounds__(256) k_dq_finalize(const float* __restrict__ dqacc, const int32_t* __restrict__ pos,
                                                     __nv_bfloat16* dq, int N, int T, int Hq, int heads_per_block,
                                                     float theta) {
  constexpr int TT = 32, HALF = HD / 2, G = HALF / 8;   // G groups of 8 columns per half row
  constexpr int PER = (HD / 4) * TT / 256;              // 16-byte loads per thread and head (256 threads)
  __shared__ float s_cos[TT][HALF], s_sin[TT][HALF];
  __shared__ float tile[HD][TT + 1];
  const int i0 = blockIdx.x * TT;
  const int h0 = blockIdx.y * heads_per_block;
  // the next head's rows are loaded into registers while the current head is rotated and
  // stored, so every thread keeps PER loads in flight through the whole block
  auto load_head = [&](int h, float4 (&v)[PER]) {
    const float* src = dqacc + ((size_t)h * T + i0 / TILE) * HD * TILE + 4 * (i0 % TILE);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = threadIdx.x + 256 * k, c4 = e / TT, t = e % TT;
      v[k] = *reinterpret_cast<const float4*>(src + ((size_t)c4 * TILE + t) * 4);
    }
  };
  float4 nxt[PER];
  load_head(h0, nxt);                                   // in flight during the angle table
  for (int e = threadIdx.x; e < TT * HALF; e += blockDim.x) {
    const int t = e / HALF, c = e % HALF;
    const int i = i0 + t;
    float sv = 0.f, cv = 1.f;
    if (theta > 0.f && i < N) sincosf(static_cast<float>(pos[i]) * rope_inv_freq(c, HD, theta), &sv, &cv);
    s_cos[t][c] = cv;
    s_sin[t][c] = sv;
  }
  const int t_out = threadIdx.x / G, g_out = threadIdx.x % G;
  for (int h = h0; h < h0 + heads_per_block; ++h) {
    __syncthreads();
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = threadIdx.x + 256 * k, c4 = e / TT, t = e % TT;
      tile[4 * c4 + 0][t] = nxt[k].x;
      tile[4 * c4 + 1][t] = nxt[k].y;
      tile[4 * c4 + 2][t] = nxt[k].z;
      tile[4 * c4 + 3][t] = nxt[k].w;
    }
    __syncthreads();
    if (h + 1 < h0 + heads_per_block) load_head(h + 1, nxt);
    const int i = i0 + t_out;
    if (t_out < TT && i < N) {
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a[2], b[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c = 8 * g_out + 2 * e + k;
          const float g1 = tile[c][t_out], g2 = tile[c + HALF][t_out];
          const float cv = s_cos[t_out][c], sv = s_sin[t_out][c];
          a[k] = g1 * cv + g2 * sv;
          b[k] = g2 * cv - g1 * sv;
        }
        lo[e] = pack_bf16(a[0], a[1]);
        hi[e] = pack_bf16(b[0], b[1]);
      }
      __nv_bfloat16* row = dq + ((size_t)i * Hq + h) * HD;
      *reinterpret_cast<uint4*>(row + 8 * g_out) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(row + HALF + 8 * g_out) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <int HD>
int launch_bwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, const tree_bf16* v,
               const tree_bf16* o, const float* lse, const tree_bf16* dO, const float* w, int Hq, int Hkv, float scale,
               float theta, void* ws, tree_bf16* dq, tree_bf16* dk, tree_bf16* dv, const tree_gateway_t* gw,
               float* dk_gw, float* dv_gw, int32_t* status, cudaStream_t s) {
  using C = BwdCfg<HD>;
  const int N = plan->n_tokens, T = plan->n_tiles, Npad = T * TILE;
  float* ndlt = static_cast<float*>(ws);
  float* nlse2 = ndlt + (size_t)Hq * Npad;
  float* dqacc = reinterpret_cast<float*>(static_cast<char*>(ws) + align256((size_t)2 * Hq * Npad * 4));
  CUtensorMap tq, tk, tv, tdo, tkg, tvg;
  int rc = make_tmap_bf16_3d(&tq, q, HD, Hq, N);
  if (!rc) rc = make_tmap_bf16_3d(&tk, k, HD, Hkv, N);
  if (!rc) rc = make_tmap_bf16_3d(&tv, v, HD, Hkv, N);
  if (!rc) rc = make_tmap_bf16_3d(&tdo, dO, HD, Hq, N);
  if (!rc && gw) rc = make_tmap_bf16_3d(&tkg, gw->k, HD, Hkv, gw->len);
  if (!rc && gw) rc = make_tmap_bf16_3d(&tvg, gw->v, HD, Hkv, gw->len);
  if (rc) return rc;
  if (!gw) { tkg = tk; tvg = tv; }              // unused without a gateway
  const int A = gw ? gw->len : 0, G = (A + TILE - 1) / TILE;
  rc = record_cuda(cudaFuncSetAttribute(k_bwd_dkdv<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC));
  if (rc) return rc;
  {
    // setmaxnreg.inc waits for registers released by other warpgroups of the CTA: the
    // re-balancing only adds up if the kernel launches with exactly LAUNCH_REGS per thread.
    cudaFuncAttributes fa;
    rc = record_cuda(cudaFuncGetAttributes(&fa, k_bwd_dkdv<HD>));
    if (rc) return rc;
    if (fa.numRegs != C::LAUNCH_REGS) {
      record_cuda(cudaErrorInvalidConfiguration);
      return TREE_ERR_CUDA;
    }
  }
  record_timing_event(0, s);
  {
    k_bwd_pre<HD><<<dim3(Npad / 32, Hq), 256, 0, s>>>(
        reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(dO), lse, w, ndlt, nlse2, scale, dqacc, N,
        Npad, Hq);
  }
  // CTAs per column: small grids split every column over a cluster (see tree_set_bwd_split)
  const int ctas = (T + G) * Hkv;
  int dev = 0, sms = 0;
  rc = record_cuda(cudaGetDevice(&dev));
  if (!rc) rc = record_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (rc) return rc;
  // Clusters are used only while the split grid still fits one wave of SMs: a cluster needs all
  // its SMs free at once, which costs throughput on a full GPU (measured: no gain at 216 CTAs
  // on 152 SMs, and a 2064-CTA gateway backward 0.51 -> 0.91 ms when forced to 2)
  int split = bwd_split_override();
  if (split == 0) {
    split = 1;
    while (split < 4 && (int64_t)ctas * split * 2 <= sms) split *= 2;   // the doubled grid fits one wave
  }
  BwdParams P{plan->col_ptr, plan->col_idx, plan->col_order, plan->tok_in, plan->tok_out, plan->pos,
              plan->tile_runs, plan->tile_nruns, plan->tile_class, nlse2, ndlt, dqacc, reinterpret_cast<__nv_bfloat16*>(dk),
              reinterpret_cast<__nv_bfloat16*>(dv), status, N, T, Npad, Hq, Hkv, Hq / Hkv, scale,
              scale * 1.4426950408889634f, theta, A, G, split, dk_gw, dv_gw, wait_limit_ns()};
  record_timing_event(1, s);
  if (split == 1) {
    k_bwd_dkdv<HD><<<ctas, C::THREADS, C::SMEM_ALLOC, s>>>(tq, tk, tv, tdo, tkg, tvg, P);
  } else {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ctas * split);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = split;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    rc = record_cuda(cudaLaunchKernelEx(&cfg, k_bwd_dkdv<HD>, tq, tk, tv, tdo, tkg, tvg, P));
    if (rc) return rc;
  }
  record_timing_event(2, s);
  {
    int hpb = 1;                                  // heads per block: the largest divisor of Hq up to 8
    for (int c = 8; c > 1; --c)
      if (Hq % c == 0) { hpb = c; break; }
    k_dq_finalize<HD><<<dim3((N + 31) / 32, Hq / hpb), 256, 0, s>>>(
        dqacc, plan->pos, reinterpret_cast<__nv_bfloat16*>(dq), N, T, Hq, hpb, theta);
  }
  record_timing_event(3, s);
  return record_cuda(cudaGetLastError());
}

}  // namespace
}  // namespace ta

using namespace ta;

extern "C" size_t tree_attn_bwd_workspace(const tree_plan_t* plan, int Hq, int d) {
  if (!plan || Hq <= 0 || d <= 0) return 0;
  const size_t Np = (size_t)plan->n_tiles * TILE;
  return align256(2 * Np * Hq * 4) + align256((size_t)Hq * d * Np * 4);
}

namespace ta {
namespace {
int bwd_entry(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, const tree_bf16* v,
              const tree_bf16* o, const float* lse, const tree_bf16* dO, const float* w, int Hq, int Hkv, int d,
              float scale, float rope_theta, void* workspace, tree_bf16* dq, tree_bf16* dk, tree_bf16* dv,
              const tree_gateway_t* gw, float* dk_gw, float* dv_gw, int32_t* status_dev, tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse || !dO || !workspace || !dq || !dk || !dv) return TREE_ERR_ARG;
  if ((d != 64 && d != 128) || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return TREE_ERR_SHAPE;
  for (const void* ptr : {(const void*)o, (const void*)dO, (const void*)dq, (const void*)dk, (const void*)dv})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return TREE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(lse) & 15)) return TREE_ERR_ARG;
  if (gw && (!gw->k || !gw->v || gw->len <= 0 || !dk_gw || !dv_gw || (reinterpret_cast<uintptr_t>(dk_gw) & 15) ||
             (reinterpret_cast<uintptr_t>(dv_gw) & 15)))
    return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  if (!(scale > 0.f)) scale = 1.f / sqrtf(static_cast<float>(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 128 ? launch_bwd<128>(plan, q, k, v, o, lse, dO, w, Hq, Hkv, scale, rope_theta, workspace, dq, dk, dv,
                                    gw, dk_gw, dv_gw, status_dev, s)
                  : launch_bwd<64>(plan, q, k, v, o, lse, dO, w, Hq, Hkv, scale, rope_theta, workspace, dq, dk, dv, gw,
                                   dk_gw, dv_gw, status_dev, s);
}

// parent rows += fp32 gateway gradients, one thread per 8 columns of a (row, kv head)
__global__ void k_relay_add(const int32_t* __restrict__ rows, int A, const float* __restrict__ gk,
                            const float* __restrict__ gv, __nv_bfloat16* dk, __nv_bfloat16* dv, int HkvD) {
  const size_t e = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (e >= (size_t)A * HkvD) return;
  const size_t r = e / HkvD, c = e % HkvD;
  const size_t dst = (size_t)rows[r] * HkvD + c;
  for (int which = 0; which < 2; ++which) {
    const float* src = (which ? gv : gk) + e;
    uint4* out = reinterpret_cast<uint4*>((which ? dv : dk) + dst);
    const uint4 cur = *out;
    const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
    *out = make_uint4(pack_bf16(bf16lo(cur.x) + a.x, bf16hi(cur.x) + a.y), pack_bf16(bf16lo(cur.y) + a.z, bf16hi(cur.y) + a.w),
                      pack_bf16(bf16lo(cur.z) + b.x, bf16hi(cur.z) + b.y), pack_bf16(bf16lo(cur.w) + b.z, bf16hi(cur.w) + b.w));
  }
}
}  // namespace
}  // namespace ta

extern "C" int tree_attn_bwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, const tree_bf16* v,
                             const tree_bf16* o, const float* lse, const tree_bf16* dO, int Hq, int Hkv, int d,
                             float scale, float rope_theta, void* workspace, tree_bf16* dq, tree_bf16* dk,
                             tree_bf16* dv, int32_t* status_dev, tree_stream_t stream) {
  return bwd_entry(plan, q, k, v, o, lse, dO, nullptr, Hq, Hkv, d, scale, rope_theta, workspace, dq, dk, dv, nullptr,
                   nullptr, nullptr, status_dev, stream);
}

extern "C" int tree_attn_bwd_weighted(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                                      const tree_bf16* v, const tree_bf16* o, const float* lse, const tree_bf16* u,
                                      int Hq, int Hkv, int d, float scale, float rope_theta, void* workspace,
                                      tree_bf16* dq, tree_bf16* dk, tree_bf16* dv, int32_t* status_dev,
                                      tree_stream_t stream) {
  if (!plan || !plan->w) return TREE_ERR_ARG;
  return bwd_entry(plan, q, k, v, o, lse, u, plan->w, Hq, Hkv, d, scale, rope_theta, workspace, dq, dk, dv, nullptr,
                   nullptr, nullptr, status_dev, stream);
}

extern "C" int tree_attn_bwd_gateway(const tree_plan_t* plan, const tree_gateway_t* gw, const tree_bf16* q,
                                     const tree_bf16* k, const tree_bf16* v, const tree_bf16* o, const float* lse,
                                     const tree_bf16* dO, int Hq, int Hkv, int d, float scale, float rope_theta,
                                     void* workspace, tree_bf16* dq, tree_bf16* dk, tree_bf16* dv, float* dk_gw,
                                     float* dv_gw, int32_t* status_dev, tree_stream_t stream) {
  if (!gw) return TREE_ERR_ARG;
  return bwd_entry(plan, q, k, v, o, lse, dO, nullptr, Hq, Hkv, d, scale, rope_theta, workspace, dq, dk, dv, gw, dk_gw,
                   dv_gw, status_dev, stream);
}

extern "C" int tree_relay_add(const int32_t* rows, int32_t len, const float* dk_gw, const float* dv_gw, int Hkv,
                              int d, tree_bf16* dk, tree_bf16* dv, tree_stream_t stream) {
  if (!rows || !dk_gw || !dv_gw || !dk || !dv || len <= 0) return TREE_ERR_ARG;
  if ((d != 64 && d != 128) || Hkv <= 0) return TREE_ERR_SHAPE;
  for (const void* ptr : {(const void*)dk_gw, (const void*)dv_gw, (const void*)dk, (const void*)dv})
    if (reinterpret_cast<uintptr_t>(ptr) & 15) return TREE_ERR_ARG;
  int rc = check_device();
  if (rc) return rc;
  const size_t groups = (size_t)len * Hkv * d / 8;
  k_relay_add<<<(unsigned)((groups + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      rows, len, dk_gw, dv_gw, reinterpret_cast<__nv_bfloat16*>(dk), reinterpret_cast<__nv_bfloat16*>(dv), Hkv * d);
  return record_cuda(cudaGetLastError());
}

// ------------------------------------------------------------------------------------------
// Non-allocating backward: the same kernels, with the delta / dQ-accumulator scratch taken
// from one fixed device array instead of a caller workspace (for callers that cannot
// allocate device memory).  The array is shared by every call on a device; the accumulator
// is zeroed at the start of each call, and overlapping calls race on it.
namespace ta {
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[TREE_NOALLOC_SCRATCH_BYTES];

// The array's device address in the current device's context.  It is looked up on every call
// (a host-side symbol lookup that allocates nothing) rather than cached: after cudaDeviceReset,
// or any other teardown of the context, the module is loaded again and the array may move.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  const int rc = record_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch));
  if (rc) return rc;
  *out = p;
  return TREE_OK;
}
}  // namespace
}  // namespace ta

extern "C" int tree_attn_bwd_noalloc(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k,
                                     const tree_bf16* v, const tree_bf16* o, const float* lse, const tree_bf16* dO,
                                     int Hq, int Hkv, int d, float scale, float rope_theta, tree_bf16* dq,
                                     tree_bf16* dk, tree_bf16* dv, int32_t* status_dev, tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if ((d != 64 && d != 128) || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return TREE_ERR_SHAPE;
  if (tree_attn_bwd_workspace(plan, Hq, d) > TREE_NOALLOC_SCRATCH_BYTES) return TREE_ERR_SCRATCH;
  rc = check_device();
  if (rc) return rc;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  return tree_attn_bwd(plan, q, k, v, o, lse, dO, Hq, Hkv, d, scale, rope_theta, scratch, dq, dk, dv, status_dev,
                       stream);
}
