// Tree-masked attention forward on tcgen05 ("Tree Training 技术详解", section 4.2:
// Softmax(Q K^T / sqrt(d) + M) V with the tree mask M; section 4.3: block-sparse over the
// ancestor tiles, mask evaluated only where a tile is partly visible).
//
// One CTA computes one query tile for NH q heads that read the same kv head (NH = 2 when the
// GQA group size is even, else 1), walking the non-empty key tiles of the tile's row.  Each
// K/V tile is loaded once for both heads.
//   warps 0, 2    TMA producers: warp 0 the NH Q tiles once, then K tiles into a 2-stage ring;
//                 warp 2 the V tiles (with the key tile's dfs_in/dfs_out words and node runs)
//                 into another.  A K stage is free as soon as every head's S MMA has read it, a
//                 V stage only after the last P V, so the next K tile starts loading a step
//                 earlier than with one ring for both;
//   warp 1        allocates TMEM and issues every tcgen05.mma from one thread, head-interleaved:
//                 O_i += P_i V(n-1), then S_i = Q_i K(n)^T, for i = 0..NH-1;
//   warps 4+4i..  softmax warpgroup i (head i): thread r owns query row r (TMEM lane r), so the
//                 row max and sum never leave the thread.  It reads S_i from TMEM, masks partial
//                 tiles with dfs_in(node j) <= dfs_in(node i) <= dfs_out(node j) (and j <= i on
//                 the diagonal tile), and writes P_i as bf16 back into the first half of S_i's
//                 TMEM columns, where the P V MMA reads it as its A operand.
// Online softmax per row, log2 units: m_ref is the offset O and l are scaled by.  It is moved
// (and O rescaled in TMEM) only when the running max exceeds it by more than 8, so every P
// value is at most 2^8; O / l is the same exact quotient whichever offset was used.  Two
// partial states relate by the associative merge of the Tree Attention page.
#include <cmath>

#include "common.cuh"

namespace ta {
namespace {

constexpr int kMaxList = 1024;      // row lists up to this length are staged in shared memory
constexpr int kGwBit = 4;           // tile class flag of a gateway tile (class in the low bits)

template <int HD, int NH>
struct FwdCfg {
  static constexpr int NCH = HD / 64;                 // 64-column (128-byte) chunks per row
  static constexpr int NS = 2;                        // K/V ring stages
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NH * NCH * CHUNK_BYTES;
  static constexpr int V_OFF = K_OFF + NS * NCH * CHUNK_BYTES;
  static constexpr int KIN_OFF = V_OFF + NS * NCH * CHUNK_BYTES;
  static constexpr int KOUT_OFF = KIN_OFF + NS * TILE * 4;
  static constexpr int RUNS_OFF = KOUT_OFF + NS * TILE * 4;    // [NS][TREE_MAX_RUNS] int4 node runs
  static constexpr int LIST_OFF = RUNS_OFF + NS * TREE_MAX_RUNS * 16;   // int32 key tiles of the row
  static constexpr int LCLS_OFF = LIST_OFF + kMaxList * 4;     // uint8 their tile classes
  static constexpr int BAR_OFF = LCLS_OFF + kMaxList;
  static constexpr int NBAR = 1 + 4 * NS + 3 * NH + 3;  // q, k and v full/empty, s/p/o per head, drain, peers
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;      // slack for 1024-byte alignment
  // warpgroup 0: K producer (warp 0), MMA issuer (warp 1), V producer (warp 2), one idle warp; then one softmax
  // warpgroup per head.  With two heads the softmax warpgroups take registers from warpgroup 0.
  static constexpr int THREADS = 128 + NH * 128;
  static constexpr int LAUNCH_REGS = 168;             // 384 x 168 = 64512 (two heads)
  static constexpr int REGS_CTRL = 88, REGS_SOFTMAX = 208;
  static_assert(NH == 1 || 128 * REGS_CTRL + 256 * REGS_SOFTMAX <= THREADS * LAUNCH_REGS,
                "register re-balancing must fit the launch allocation");
  // TMEM: S_i at columns 128 i (P_i packed bf16 in its first 64), O_i at 128 NH + HD i
  static constexpr uint32_t O_COL0 = 128 * NH;
  static constexpr uint32_t TMEM_NEED = 128 * NH + HD * NH;
  static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
  static constexpr uint32_t IDESC_S = idesc_bf16(TILE, TILE, 0, 0);   // Q K-major, K K-major
  static constexpr uint32_t IDESC_PV = idesc_bf16(TILE, HD, 0, 1);    // P (TMEM) K-major, V MN-major
  static constexpr uint32_t K_TX = NCH * CHUNK_BYTES;
  static constexpr uint32_t V_TX = NCH * CHUNK_BYTES + 2 * TILE * 4 + TREE_MAX_RUNS * 16;   // V + mask data
  static constexpr uint32_t VG_TX = NCH * CHUNK_BYTES;                // a gateway tile: V only
  static constexpr float RESCALE_THRESHOLD = 8.f;     // log2 units
  // split rows: a CTA of rank > 0 leaves its per-row softmax state (O row scaled by 2^-m_ref,
  // then m_ref and l) here after its main loop, over the Q and K / V buffers, free by then
  static constexpr int PART_ROW = HD + 4;
  static constexpr int PART_OFF = 0;
  static constexpr int PART_BYTES = NH * TILE * PART_ROW * 4;
  static_assert(PART_OFF + PART_BYTES <= KIN_OFF, "partial-state area must stay below the mask data");
};

struct FwdParams {
  const int32_t* row_ptr;
  const int32_t* row_idx;
  const int32_t* row_order;
  const int32_t* tok_in;
  const int32_t* tok_out;
  const int32_t* tile_runs;
  const int32_t* tile_nruns;
  const uint8_t* tile_class;
  __nv_bfloat16* o;
  float* lse;
  int32_t* status;
  int N, T, Npad, Hq, grp, n_hgroups;
  int gw_len, gw_tiles;      // gateway prefix: keys every query sees (0 = none), its 128-key tiles
  int split;                 // CTAs per row (a cluster): CTA s takes the row's tiles s, s + split, ...
  float scale_log2;          // softmax scale * log2(e)
  uint64_t wait_ns;
};

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

// GW: the instantiation with gateway tiles in front of each row (the plain tree keeps the
// code without the gateway branches)
template <int HD, int NH, bool GW>
__global__ void __launch_bounds__(FwdCfg<HD, NH>::THREADS, 1)
    k_attn_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKg,
               const __grid_constant__ CUtensorMap tmVg, const FwdParams p) {
  using C = FwdCfg<HD, NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 1 + C::NS;
  uint64_t* v_full = bars + 1 + 2 * C::NS;            // V tile with the key tile's mask data
  uint64_t* v_empty = bars + 1 + 3 * C::NS;
  uint64_t* s_full = bars + 1 + 4 * C::NS;            // [NH] S_i(n) computed (and PV_i(n-1) done)
  uint64_t* p_full = s_full + NH;                     // [NH] P_i(n) in TMEM, O_i rescaled
  uint64_t* o_done = p_full + NH;                     // [NH] last PV_i done
  uint64_t* drain = o_done + NH;
  uint64_t* peer_ready = drain + 1;                   // rank 0: the other ranks' row states are in place
  uint64_t* peer_done = drain + 2;                    // rank > 0: rank 0 has read this CTA's states
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  int* abort_flag = reinterpret_cast<int*>(sm + C::MISC_OFF + 4);
  int32_t* kin_s = reinterpret_cast<int32_t*>(sm + C::KIN_OFF);
  int32_t* kout_s = reinterpret_cast<int32_t*>(sm + C::KOUT_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // clusters of p.split CTAs share one row: rank s takes the row's tiles s, s + split, ...; their
  // softmax states are merged at the end (the associative (max, numerator, denominator) merge)
  const int srank = p.split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int u = blockIdx.x / p.split;
  const int qt = p.row_order[u / p.n_hgroups];
  const int h0 = (u % p.n_hgroups) * NH;              // first q head of this CTA
  const int kvh = h0 / p.grp;
  const int rp0 = p.row_ptr[qt];
  const int rcnt = p.row_ptr[qt + 1] - rp0;
  const int G = GW ? p.gw_tiles : 0;
  const int cnt_all = G + rcnt;                       // gateway tiles first, then the row's own
  const int cnt = cnt_all > srank ? (cnt_all - srank + p.split - 1) / p.split : 0;   // this CTA's
  int32_t* list_s = reinterpret_cast<int32_t*>(sm + C::LIST_OFF);
  uint8_t* lcls_s = sm + C::LCLS_OFF;
  // this CTA's tiles of the row (gateway tiles first), in its order, as key tile and class:
  // global tile n of the row is gateway tile n < G (every key before gw_len visible; the last
  // one partial when gw_len is not a multiple of 128), else the row's own tile n - G
  auto global_tile = [&](int n, int& kt, int& cls) {
    if (GW && n < G) { kt = n; cls = kGwBit | ((n == G - 1 && (p.gw_len % TILE) != 0) ? 1 : 2); return; }
    kt = p.row_idx[rp0 + n - G];
    cls = p.tile_class[(size_t)qt * p.T + kt];
  };
  for (int m = threadIdx.x; m < cnt && m < kMaxList; m += blockDim.x) {   // staged once
    int kt, cls;
    global_tile(srank + m * p.split, kt, cls);
    list_s[m] = kt;
    lcls_s[m] = static_cast<uint8_t>(cls);
  }
  auto row_tile = [&](int m, int& kt, int& cls) {     // this CTA's tile m
    if (m < kMaxList) { kt = list_s[m]; cls = lcls_s[m]; }
    else global_tile(srank + m * p.split, kt, cls);
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < NH; ++i) { mbar_init(&s_full[i], 1); mbar_init(&p_full[i], 4); mbar_init(&o_done[i], 1); }
    mbar_init(drain, 1);
    mbar_init(peer_ready, p.split > 1 ? p.split - 1 : 1);
    mbar_init(peer_done, 1);
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
  if (p.split > 1) cluster_sync_all();                // every CTA's barriers initialised before remote arrivals
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.wait_ns};

  if (warp < 4) {
    if constexpr (NH == 2) regs_dec<C::REGS_CTRL>();
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer: Q, K
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      if (GW) prefetch_tmap(&tmKg);
      // a CTA without tiles (a split row shorter than the cluster) loads nothing: its shared
      // memory then holds only the zero state it leaves for rank 0
      if (cnt > 0) {
        mbar_expect_tx(q_full, NH * C::NCH * CHUNK_BYTES);
        for (int i = 0; i < NH; ++i)
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sm + C::Q_OFF + (i * C::NCH + c) * CHUNK_BYTES, &tmQ, q_full, c * 64, h0 + i, qt * TILE);
      }
      // K(n) waits only for the S MMAs of tile n-2 (k_empty), not for its P V MMAs
      int issued = 0;
      for (int n = 0; n < cnt; ++n) {
        const int s = n % C::NS;
        int kt, cls;
        row_tile(n, kt, cls);
        if (n >= C::NS && !mbar_wait(&k_empty[s], ((n / C::NS) - 1) & 1, wc)) break;
        mbar_expect_tx(&k_full[s], C::K_TX);
        for (int c = 0; c < C::NCH; ++c)          // gateway tile rows past gw_len read as 0
          tma_load_3d(sm + C::K_OFF + (s * C::NCH + c) * CHUNK_BYTES, (GW && (cls & kGwBit)) ? &tmKg : &tmK, &k_full[s],
                      c * 64, kvh, kt * TILE);
        issued = n + 1;
      }
      if (*abort_flag) {                       // let copies in flight land before exit
        if (cnt > 0) mbar_wait_drain(q_full, 0, p.wait_ns);
        for (int n = (issued > C::NS ? issued - C::NS : 0); n < issued; ++n)
          mbar_wait_drain(&k_full[n % C::NS], (n / C::NS) & 1, p.wait_ns);
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- TMA producer: V + mask data
    if (lane == 0) {
      prefetch_tmap(&tmV);
      if (GW) prefetch_tmap(&tmVg);
      int issued = 0;
      for (int n = 0; n < cnt; ++n) {
        const int s = n % C::NS;
        int kt, cls;
        row_tile(n, kt, cls);
        const bool gwt = GW && (cls & kGwBit);
        if (n >= C::NS && !mbar_wait(&v_empty[s], ((n / C::NS) - 1) & 1, wc)) break;
        mbar_expect_tx(&v_full[s], gwt ? C::VG_TX : C::V_TX);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sm + C::V_OFF + (s * C::NCH + c) * CHUNK_BYTES, gwt ? &tmVg : &tmV, &v_full[s], c * 64, kvh,
                      kt * TILE);
        if (!gwt) {
          bulk_load(kin_s + s * TILE, p.tok_in + (size_t)kt * TILE, TILE * 4, &v_full[s]);
          bulk_load(kout_s + s * TILE, p.tok_out + (size_t)kt * TILE, TILE * 4, &v_full[s]);
          bulk_load(sm + C::RUNS_OFF + s * TREE_MAX_RUNS * 16, p.tile_runs + (size_t)kt * TREE_MAX_RUNS * 4,
                    TREE_MAX_RUNS * 16, &v_full[s]);
        }
        issued = n + 1;
      }
      if (*abort_flag)
        for (int n = (issued > C::NS ? issued - C::NS : 0); n < issued; ++n)
          mbar_wait_drain(&v_full[n % C::NS], (n / C::NS) & 1, p.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto issue_s = [&](int i, int s) {       // S_i = Q_i K(s)^T into TMEM columns 128 i
        const uint32_t q_base = smem_u32(sm + C::Q_OFF + i * C::NCH * CHUNK_BYTES);
        const uint32_t k_base = smem_u32(sm + C::K_OFF + s * C::NCH * CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK_BYTES + (kk & 3) * 32;   // d along K, 32 B per step
          umma_bf16(tmem + 128 * i, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024),
                    C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[i]);
      };
      auto issue_pv = [&](int i, int m) -> bool {   // O_i += P_i(m) V(m)
        if (!mbar_wait(&p_full[i], m & 1, wc)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sm + C::V_OFF + (m % C::NS) * C::NCH * CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)     // 16 keys per step: 8 TMEM columns of P, 16 V rows
          umma_bf16_tmem_a(tmem + C::O_COL0 + HD * i, tmem + 128 * i + kk * 8,
                           sdesc_sw128(v_base + kk * 16 * 128, CHUNK_BYTES, 1024), C::IDESC_PV,
                           (m > 0 || kk > 0) ? 1u : 0u);
        return true;
      };
      bool ok = cnt == 0 || (mbar_wait(q_full, 0, wc) && mbar_wait(&k_full[0], 0, wc));
      if (ok && cnt > 0) {
        tc_fence_after();
        for (int i = 0; i < NH; ++i) issue_s(i, 0);
        umma_commit(&k_empty[0]);
      }
      for (int n = 1; ok && n < cnt; ++n) {
        const int s = n % C::NS;
        // V(n-1) for the P V MMAs below (loaded behind K(n-1)), then K(n) for the S MMAs
        if (!mbar_wait(&v_full[(n - 1) % C::NS], ((n - 1) / C::NS) & 1, wc) ||
            !mbar_wait(&k_full[s], (n / C::NS) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        for (int i = 0; ok && i < NH; ++i) {
          if (!issue_pv(i, n - 1)) { ok = false; break; }
          if (i == NH - 1) umma_commit(&v_empty[(n - 1) % C::NS]);
          issue_s(i, s);                       // overwrites S_i / P_i: ordered after PV_i(n-1)
        }
        if (ok) umma_commit(&k_empty[s]);
      }
      if (ok && cnt > 0) ok = mbar_wait(&v_full[(cnt - 1) % C::NS], ((cnt - 1) / C::NS) & 1, wc);
      if (ok && cnt > 0) {
        for (int i = 0; ok && i < NH; ++i) {
          if (!issue_pv(i, cnt - 1)) { ok = false; break; }
          umma_commit(&o_done[i]);
        }
        umma_commit(&v_empty[(cnt - 1) % C::NS]);
      }
      umma_commit(drain);                      // completes once every MMA above is done
      mbar_wait_drain(drain, 0, p.wait_ns);
    }
  }
  } else {
    if constexpr (NH == 2) regs_inc<C::REGS_SOFTMAX>();
    // ---------------------------------------------------------------- softmax warpgroups
    const int wg = (warp - 4) >> 2;            // head index inside the CTA
    const int wq = warp & 3;                   // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;              // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + 128 * wg;
    const uint32_t o_addr = tmem + lane_off + C::O_COL0 + HD * wg;
    const int h = h0 + wg;
    const int qi = qt * TILE + r;
    const int qin = p.tok_in[qi];
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    float m_run = -INFINITY;                   // running row max (log2 units)
    float m_ref = 0.f;                         // offset O and l are currently scaled by
    float l_run = 0.f;
    bool ok = true;
    // node-run count of the tile after the current one, loaded a tile ahead so that a partial
    // tile's mask does not wait for global memory
    auto runs_of = [&](int m) -> int {
      if (m >= cnt) return 0;
      int kt, cls;
      row_tile(m, kt, cls);
      return (GW && (cls & kGwBit)) ? 0 : p.tile_nruns[kt];
    };
    int nr_next = runs_of(0);
    for (int n = 0; n < cnt; ++n) {
      const int s = n % C::NS;
      int kt, cls;
      row_tile(n, kt, cls);
      const int nr_cur = nr_next;
      nr_next = runs_of(n + 1);
      if (!mbar_wait_warp(&s_full[wg], n & 1, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[TILE];
      tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(sv + 0));
      tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(sv + 64));
      tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(sv + 96));
      tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(sv + 0));
      tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(sv + 64));
      tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(sv + 96));
      if (GW && cls == (kGwBit | 1)) {         // ragged last gateway tile: keys past gw_len
        uint32_t vm[4] = {0u, 0u, 0u, 0u};
        set_bits(vm, 0, p.gw_len - kt * TILE);
        const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
        for (int c = 0; c < TILE; ++c)
          if (!((vm[c >> 5] >> (c & 31)) & 1u)) sv[c] = ninf;
      } else if (cls == 1) {                   // partial tile: tree mask in registers
        // the key tile's mask data arrive with its V tile; that stage is refilled only after
        // the last P V of this tile, which waits for this warpgroup's P
        if (!mbar_wait_warp(&v_full[s], (n / C::NS) & 1, wc)) { ok = false; break; }
        const int nr = nr_cur;
        const int jrel = qi - kt * TILE;       // key c is causal-visible iff c <= jrel
        uint32_t vm[4] = {0u, 0u, 0u, 0u};     // bit c: key c visible to this row
        if (nr <= TREE_MAX_RUNS) {             // one ancestor-interval test per node run
          const int4* runs = reinterpret_cast<const int4*>(sm + C::RUNS_OFF + s * TREE_MAX_RUNS * 16);
          for (int k = 0; k < nr; ++k) {
            const int4 rn = runs[k];
            if (rn.z <= qin && qin <= rn.w) set_bits(vm, rn.x, rn.y);
          }
        } else {                               // many tiny nodes: test every key
          const int4* kin4 = reinterpret_cast<const int4*>(kin_s + s * TILE);
          const int4* kout4 = reinterpret_cast<const int4*>(kout_s + s * TILE);
          for (int c4 = 0; c4 < TILE / 4; ++c4) {
            const int4 a = kin4[c4], z = kout4[c4];
            const uint32_t bits = (uint32_t)(a.x <= qin && qin <= z.x) | ((uint32_t)(a.y <= qin && qin <= z.y) << 1) |
                                  ((uint32_t)(a.z <= qin && qin <= z.z) << 2) | ((uint32_t)(a.w <= qin && qin <= z.w) << 3);
            vm[c4 >> 3] |= bits << (4 * (c4 & 7));
          }
        }
        set_bits_clear_above(vm, jrel);        // causal: keep keys c <= jrel
        const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
        for (int c = 0; c < TILE; ++c)
          if (!((vm[c >> 5] >> (c & 31)) & 1u)) sv[c] = ninf;
      }
      float mx[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e] = fmaxf(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]));
#pragma unroll
      for (int c = 8; c < TILE; c += 8)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx[e] = fmax3(mx[e], __uint_as_float(sv[c + 2 * e]), __uint_as_float(sv[c + 2 * e + 1]));
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float m_new = fmaxf(m_run, mt * sl2);
      m_run = m_new;
      float alpha = 1.f;
      if (l_run == 0.f) {                      // nothing accumulated yet: take the offset as is
        m_ref = (m_new == -INFINITY) ? 0.f : m_new;
      } else if (m_new > m_ref + C::RESCALE_THRESHOLD) {
        alpha = ex2_approx(m_ref - m_new);
        m_ref = m_new;
      }
      const uint64_t negm = f2_pack(-m_ref, -m_ref);
      uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
      // P_i over the first 64 columns of S_i (S_i is already in registers): 64 scores per half
#pragma unroll
      for (int q16 = 0; q16 < 8; ++q16) {        // 16 keys -> 8 packed columns at a time
        uint32_t pk[8];
#pragma unroll
        for (int c = 16 * q16; c < 16 * q16 + 16; c += 4) {
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, negm), x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2x2, negm), x2, x3);
          const float e0 = ex2_approx(x0), e1 = ex2_approx(x1), e2 = ex2_approx(x2), e3 = ex2_approx(x3);
          acc0 = f2_add(acc0, f2_pack(e0, e1));
          acc1 = f2_add(acc1, f2_pack(e2, e3));
          pk[(c - 16 * q16) >> 1] = pack_bf16(e0, e1);
          pk[((c - 16 * q16) >> 1) + 1] = pack_bf16(e2, e3);
        }
        tmem_store8(s_addr + 8 * q16, pk);
      }
      float a0, a1, a2, a3;
      f2_unpack(acc0, a0, a1);
      f2_unpack(acc1, a2, a3);
      l_run = l_run * alpha + ((a0 + a1) + (a2 + a3));
      // S_i(n) complete implies PV_i(n-1) complete: O_i is stable here
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        const uint64_t al = f2_pack(alpha, alpha);
#pragma unroll 1
        for (int j = 0; j < HD / 32; ++j) {
          uint32_t rr[32];
          tmem_load32(o_addr + j * 32, rr);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float y0, y1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(rr[c]), __uint_as_float(rr[c + 1])), al), y0, y1);
            rr[c] = __float_as_uint(y0);
            rr[c + 1] = __float_as_uint(y1);
          }
          tmem_store32(o_addr + j * 32, rr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[wg]);                 // one arrival per warp
    }
    // ---------------------------------------------------------- epilogue: O, LSE of row r
    // With split rows the cluster's ranks > 0 leave their (m_ref, l, O) here and rank 0 merges
    // them with its own by the associative rule: m = max m_q, l = sum l_q 2^(m_q - m),
    // O = sum O_q 2^(m_q - m); the output is O / l and LSE = m + log2 l (natural log on store).
    const bool have = ok && cnt > 0 && mbar_wait_warp(&o_done[wg], 0, wc);
    if (have) tc_fence_after();
    const uint32_t part_row = smem_u32(sm + C::PART_OFF) + static_cast<uint32_t>((wg * TILE + r) * C::PART_ROW * 4);
    if (p.split > 1 && srank > 0) {
      const uint32_t keep = have ? 0xffffffffu : 0u;  // a rank without tiles contributes l = 0
#pragma unroll 1
      for (int j = 0; j < HD / 32; ++j) {
        uint32_t rr[32];
        tmem_load32(o_addr + j * 32, rr);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          st_shared_v4(part_row + (32 * j + 4 * v) * 4, rr[4 * v] & keep, rr[4 * v + 1] & keep, rr[4 * v + 2] & keep,
                       rr[4 * v + 3] & keep);
      }
      st_shared_v4(part_row + HD * 4, __float_as_uint(m_ref) & keep, __float_as_uint(l_run) & keep, 0u, 0u);
      named_bar_sync(2, NH * 128);                     // every softmax thread's row is in place
      if (threadIdx.x == 128) mbar_arrive_remote(mapa_shared(smem_u32(peer_ready), 0));
      (void)mbar_wait_cluster(peer_done, 0, wc);       // rank 0 reads this area until it arrives here
    } else {
      int nsum = 1;                                    // ranks merged: this one, then 1 .. split-1
      if (p.split > 1) nsum = __all_sync(0xffffffffu, mbar_wait_cluster(peer_ready, 0, wc)) ? p.split : 1;
      float wq[4] = {1.f, 0.f, 0.f, 0.f};              // each rank's weight 2^(m_q - m)
      float L = have ? l_run : 0.f, M = m_ref;
      if (nsum > 1) {
        float mq[4], lq[4];
        mq[0] = m_ref;
        lq[0] = have ? l_run : 0.f;
#pragma unroll
        for (int q = 1; q < 4; ++q) {
          mq[q] = 0.f;
          lq[q] = 0.f;
          if (q < nsum) {
            const float4 t = ld_dsmem_f4(mapa_shared(part_row + HD * 4, static_cast<uint32_t>(q)));
            mq[q] = t.x;
            lq[q] = t.y;
          }
        }
        M = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (lq[q] > 0.f) M = fmaxf(M, mq[q]);
        L = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          wq[q] = lq[q] > 0.f ? ex2_approx(mq[q] - M) : 0.f;
          L += lq[q] * wq[q];
        }
      }
      if (have || nsum > 1) {
        const float inv_l = L > 0.f ? 1.f / L : 0.f;
        __nv_bfloat16* orow = p.o + ((size_t)qi * p.Hq + h) * HD;
#pragma unroll 1
        for (int j = 0; j < HD / 32; ++j) {
          uint32_t rr[32];
          tmem_load32(o_addr + j * 32, rr);
          float of[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) of[c] = have ? __uint_as_float(rr[c]) * wq[0] : 0.f;
#pragma unroll
          for (int q = 1; q < 4; ++q) {
            if (q < nsum && wq[q] != 0.f) {
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float4 t = ld_dsmem_f4(mapa_shared(part_row + (32 * j + 4 * v) * 4, static_cast<uint32_t>(q)));
                of[4 * v] += t.x * wq[q];
                of[4 * v + 1] += t.y * wq[q];
                of[4 * v + 2] += t.z * wq[q];
                of[4 * v + 3] += t.w * wq[q];
              }
            }
          }
          if (qi < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + j * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int c = v * 8;
              dst[v] = make_uint4(pack_bf16(of[c + 0] * inv_l, of[c + 1] * inv_l), pack_bf16(of[c + 2] * inv_l, of[c + 3] * inv_l),
                                  pack_bf16(of[c + 4] * inv_l, of[c + 5] * inv_l), pack_bf16(of[c + 6] * inv_l, of[c + 7] * inv_l));
            }
          }
        }
        p.lse[(size_t)h * p.Npad + qi] = (qi < p.N && L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : 0.f;
      }
      if (p.split > 1) {
        named_bar_sync(2, NH * 128);                   // every thread has read the other ranks' areas
        if (threadIdx.x == 128)
          for (int q = 1; q < p.split; ++q) mbar_arrive_remote(mapa_shared(smem_u32(peer_done), q));
      }
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

template <int HD, int NH, bool GW>
int launch_fwd(const tree_plan_t* plan, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tkg, const CUtensorMap& tvg, int gw_len, int Hq, int Hkv, float scale, tree_bf16* o,
               float* lse, int32_t* status, cudaStream_t s) {
  using C = FwdCfg<HD, NH>;
  const int N = plan->n_tokens, T = plan->n_tiles;
  int rc = record_cuda(
      cudaFuncSetAttribute(k_attn_fwd<HD, NH, GW>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC));
  if (rc) return rc;
  // CTAs per row: split only while the split grid still fits one wave of SMs (a cluster needs
  // all its SMs free at once); rows then go to clusters whose states merge at the end.
  // Measured: a 256-token partition below a 32K-token gateway (32 CTAs) 444 -> 174 us at 4.
  const int ctas = T * (Hq / NH);
  int split = fwd_split_override();
  if (split == 0) {
    int dev = 0, sms = 0;
    rc = record_cuda(cudaGetDevice(&dev));
    if (!rc) rc = record_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (rc) return rc;
    split = 1;
    while (split < 4 && (int64_t)ctas * split * 2 <= sms) split *= 2;   // the doubled grid fits one wave
  }
  FwdParams P{plan->row_ptr, plan->row_idx, plan->row_order, plan->tok_in, plan->tok_out, plan->tile_runs,
              plan->tile_nruns, plan->tile_class,
              reinterpret_cast<__nv_bfloat16*>(o), lse, status, N, T, T * TILE, Hq, Hq / Hkv, Hq / NH,
              gw_len, (gw_len + TILE - 1) / TILE, split, scale * 1.4426950408889634f, wait_limit_ns()};
  if constexpr (NH == 2) {
    // setmaxnreg.inc waits for registers the other warpgroups released: the re-balancing only
    // adds up if the kernel launches with exactly LAUNCH_REGS per thread.
    cudaFuncAttributes fa;
    rc = record_cuda(cudaFuncGetAttributes(&fa, k_attn_fwd<HD, NH, GW>));
    if (rc) return rc;
    if (fa.numRegs != C::LAUNCH_REGS) {
      record_cuda(cudaErrorInvalidConfiguration);
      return TREE_ERR_CUDA;
    }
  }
  if (split == 1) {
    k_attn_fwd<HD, NH, GW><<<ctas, C::THREADS, C::SMEM_ALLOC, s>>>(tq, tk, tv, tkg, tvg, P);
    return record_cuda(cudaGetLastError());
  }
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
  return record_cuda(cudaLaunchKernelEx(&cfg, k_attn_fwd<HD, NH, GW>, tq, tk, tv, tkg, tvg, P));
}

}  // namespace
}  // namespace ta

using namespace ta;

namespace ta {
namespace {
int fwd_entry(const tree_plan_t* plan, const tree_gateway_t* gw, const tree_bf16* q, const tree_bf16* k,
              const tree_bf16* v, int Hq, int Hkv, int d, float scale, tree_bf16* o, float* lse, int32_t* status_dev,
              tree_stream_t stream) {
  int rc = plan_ok(plan);
  if (rc) return rc;
  if (!q || !k || !v || !o || !lse) return TREE_ERR_ARG;
  if ((d != 64 && d != 128) || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return TREE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(o) & 15) || (reinterpret_cast<uintptr_t>(lse) & 3)) return TREE_ERR_ARG;
  if (gw && (!gw->k || !gw->v || gw->len <= 0)) return TREE_ERR_ARG;
  rc = check_device();
  if (rc) return rc;
  if (!(scale > 0.f)) scale = 1.f / sqrtf(static_cast<float>(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int N = plan->n_tokens;
  CUtensorMap tq, tk, tv, tkg, tvg;
  rc = make_tmap_bf16_3d(&tq, q, d, Hq, N);
  if (!rc) rc = make_tmap_bf16_3d(&tk, k, d, Hkv, N);
  if (!rc) rc = make_tmap_bf16_3d(&tv, v, d, Hkv, N);
  if (!rc && gw) rc = make_tmap_bf16_3d(&tkg, gw->k, d, Hkv, gw->len);
  if (!rc && gw) rc = make_tmap_bf16_3d(&tvg, gw->v, d, Hkv, gw->len);
  if (rc) return rc;
  if (!gw) { tkg = tk; tvg = tv; }              // unused without a gateway
  const int A = gw ? gw->len : 0;
  const bool pair = ((Hq / Hkv) % 2) == 0;   // two q heads of one kv group per CTA
  if (gw) {
    if (d == 128)
      return pair ? launch_fwd<128, 2, true>(plan, tq, tk, tv, tkg, tvg, A, Hq, Hkv, scale, o, lse, status_dev, s)
                  : launch_fwd<128, 1, true>(plan, tq, tk, tv, tkg, tvg, A, Hq, Hkv, scale, o, lse, status_dev, s);
    return pair ? launch_fwd<64, 2, true>(plan, tq, tk, tv, tkg, tvg, A, Hq, Hkv, scale, o, lse, status_dev, s)
                : launch_fwd<64, 1, true>(plan, tq, tk, tv, tkg, tvg, A, Hq, Hkv, scale, o, lse, status_dev, s);
  }
  if (d == 128)
    return pair ? launch_fwd<128, 2, false>(plan, tq, tk, tv, tkg, tvg, 0, Hq, Hkv, scale, o, lse, status_dev, s)
                : launch_fwd<128, 1, false>(plan, tq, tk, tv, tkg, tvg, 0, Hq, Hkv, scale, o, lse, status_dev, s);
  return pair ? launch_fwd<64, 2, false>(plan, tq, tk, tv, tkg, tvg, 0, Hq, Hkv, scale, o, lse, status_dev, s)
              : launch_fwd<64, 1, false>(plan, tq, tk, tv, tkg, tvg, 0, Hq, Hkv, scale, o, lse, status_dev, s);
}
}  // namespace
}  // namespace ta

extern "C" int tree_attn_fwd(const tree_plan_t* plan, const tree_bf16* q, const tree_bf16* k, const tree_bf16* v,
                             int Hq, int Hkv, int d, float scale, tree_bf16* o, float* lse, int32_t* status_dev,
                             tree_stream_t stream) {
  return fwd_entry(plan, nullptr, q, k, v, Hq, Hkv, d, scale, o, lse, status_dev, stream);
}

extern "C" int tree_attn_fwd_gateway(const tree_plan_t* plan, const tree_gateway_t* gw, const tree_bf16* q,
                                     const tree_bf16* k, const tree_bf16* v, int Hq, int Hkv, int d, float scale,
                                     tree_bf16* o, float* lse, int32_t* status_dev, tree_stream_t stream) {
  if (!gw) return TREE_ERR_ARG;
  return fwd_entry(plan, gw, q, k, v, Hq, Hkv, d, scale, o, lse, status_dev, stream);
}
