// Device primitives for sm_103a: mbarriers with bounded waits, TMA bulk/tensor copies,
// tcgen05 (UMMA issue, commit, TMEM alloc/load/store) and shared-memory descriptors.
// All PTX here is hand-written against the public PTX ISA (tcgen05, cp.async.bulk, mbarrier).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tree_attn.h"

#define DEVI __device__ __forceinline__

namespace ta {

constexpr int TILE = TREE_TILE;
constexpr int CHUNK_BYTES = TILE * 128;      // one 128-row x 128-byte swizzled box = 16 KiB

// ------------------------------------------------------------------------------------------
// generic helpers
DEVI uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

DEVI uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

DEVI float ex2_approx(float x) {   // hardware 2^x (MUFU), -inf -> +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

DEVI uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

DEVI float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
DEVI float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// packed fp32 pairs (sm_100+ f32x2 arithmetic) and 3-input max
DEVI uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
DEVI void f2_unpack(uint64_t v, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v)); }
DEVI uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
DEVI uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DEVI uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DEVI float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ------------------------------------------------------------------------------------------
// mbarrier
DEVI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
DEVI void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
DEVI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared state of the bounded waits of one CTA: the first waiter that runs out of time
// stores TREE_ERR_TIMEOUT to the global status word and raises the CTA-wide abort flag;
// every other wait then gives up at once.
struct WaitCtl {
  volatile int* abort_flag;   // shared memory
  int32_t* status;            // global, may be null
  uint64_t limit_ns;
};

DEVI bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*wc.abort_flag) return false;
      if (global_timer_ns() - t0 > wc.limit_ns) {
        *wc.abort_flag = 1;
        if (wc.status) atomicExch(wc.status, TREE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-collective form for warps that go on to tcgen05.ld/st (.sync.aligned: every lane must
// execute them together).  All lanes wait, then agree: if any lane gave up, all do, and the
// warp leaves convergent either way.
DEVI bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
  const bool ok = mbar_wait(bar, parity, wc);
  return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------------------------------------
// thread-block clusters (distributed shared memory)
DEVI uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared-memory location in CTA `rank` of the cluster
DEVI uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// every thread of every CTA of the cluster (a hardware barrier, like __syncthreads)
DEVI void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// arrive once on an mbarrier of another CTA of the cluster; the calling thread's earlier
// writes (and those ordered before them) are released at cluster scope
DEVI void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
DEVI bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
DEVI void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
DEVI float4 ld_dsmem_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

// The same bounded wait with cluster-scope acquire: for barriers that other CTAs of the
// cluster arrive on (their released writes are visible after it returns true).
DEVI bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*wc.abort_flag) return false;
      if (global_timer_ns() - t0 > wc.limit_ns) {
        *wc.abort_flag = 1;
        if (wc.status) atomicExch(wc.status, TREE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// v[e] += the CNT fp32 values at shared offset `saddr` of cluster ranks 1 .. nsum-1, in rank order
template <int CNT>
DEVI void add_cluster_partials(float (&v)[CNT], uint32_t saddr, int nsum) {
  for (int q = 1; q < nsum; ++q) {
#pragma unroll
    for (int e = 0; e < CNT; e += 4) {
      const float4 t = ld_dsmem_f4(mapa_shared(saddr + 4 * e, static_cast<uint32_t>(q)));
      v[e] += t.x;
      v[e + 1] += t.y;
      v[e + 2] += t.z;
      v[e + 3] += t.w;
    }
  }
}

// ------------------------------------------------------------------------------------------
// TMA
DEVI void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
DEVI void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
DEVI void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// make this thread's generic-proxy shared-memory writes visible to the async proxy (UMMA)
DEVI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// element-wise atomic add of a shared-memory box into global memory through a 2-D tensor map
// (the box layout in shared memory is row-major, unswizzled); completion via bulk groups
// global[0, bytes) += shared[0, bytes) in fp32, performed by the TMA unit (16-byte aligned,
// bytes a multiple of 16); completion tracked by the bulk groups of the issuing thread
DEVI void bulk_reduce_add_f32(float* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
DEVI void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until the shared-memory sources of every committed bulk group but the newest have been read
DEVI void bulk_wait_group_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// ... all but the two newest
DEVI void bulk_wait_group_read2() { asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); }
// wait until every committed bulk group has completed (its global writes performed)
DEVI void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
DEVI void named_bar_sync(int id, int count) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory"); }
// named barrier that also returns the AND of `pred` over the `count` participating threads
DEVI bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Per-warpgroup register re-balancing (all four warps of a warpgroup execute it together).
template <int N>
DEVI void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
DEVI void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

// ------------------------------------------------------------------------------------------
// tcgen05
DEVI void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
DEVI void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {    // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate), issued by one thread
DEVI void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with the A operand read from TMEM (K-major: lane = row m, two bf16 per 32-bit column,
// the even k in the low half); a_tmem addresses the first column of this K-step's 8 columns.
DEVI void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive (once) on `bar` when every tcgen05 op this thread issued so far has completed
DEVI void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, dense, no negation.
// a_mn / b_mn select MN-major (1) or K-major (0) operands.  N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor with 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B into 1024-byte aligned boxes of 128-byte rows).
//   K-major operand : rows of 128 B along K, 8-row groups SBO apart (LBO unused);
//   MN-major operand: rows of 128 B along MN indexed by K, 8-row K groups SBO apart,
//                     64-element MN blocks LBO apart.
DEVI uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;     // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;     // swizzle mode: 128 B
  return d;
}

// The same descriptor for an address `bytes` further on (the start address field holds
// address / 16 in 14 bits: shared-memory addresses below 256 KiB never carry out of it).
DEVI uint64_t sdesc_adv(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// TMEM loads/stores, 32 data-path lanes x 32 bits, 32 consecutive columns per thread.
// The register array is tied to the wait so that no use is scheduled before it.
DEVI void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
DEVI void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
DEVI void tmem_load32(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
  tmem_wait_ld(r);
}
DEVI void tmem_store32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
DEVI void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16-column forms of the above
DEVI void tmem_load16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}
DEVI void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {    // issue only; pair with tmem_wait_ld16
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// waits for every tcgen05.ld of this thread issued so far; ties the register set to the wait
DEVI void tmem_wait_ld16(uint32_t (&a)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15])
               :
               : "memory");
}
// waits for every tcgen05.ld of this thread issued so far; ties both register sets to the wait
DEVI void tmem_wait_ld16x2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}
DEVI void tmem_store8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Store 8 bf16 (one 16-byte unit u of a 128-byte row) into a 128B-swizzled K-major box.
DEVI void st_swizzled_unit(uint8_t* box, int row, int unit, uint4 v) {
  const int phys = unit ^ (row & 7);
  *reinterpret_cast<uint4*>(box + row * 128 + phys * 16) = v;
}

// Visibility bits of a 128-key (or 128-query) tile from its node runs: run k covers tile
// columns [start, end) and is visible when its node interval contains `x`
// (dfs_in(run) <= x <= dfs_out(run), the ancestor test on DFS intervals); with `inner` the
// roles swap: the run's node must lie inside [x_lo, x_hi].
DEVI void set_bits(uint32_t (&m)[4], int a, int b) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int lo = max(a, 32 * w) - 32 * w, hi = min(b, 32 * w + 32) - 32 * w;
    if (lo < hi) m[w] |= (hi - lo == 32) ? 0xffffffffu : (((1u << (hi - lo)) - 1u) << lo);
  }
}

// keep only bits c <= j (j < 0: none, j >= 127: all)
DEVI void set_bits_clear_above(uint32_t (&m)[4], int j) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int t = j - 32 * w;                  // highest kept bit inside word w
    m[w] &= (t >= 31) ? 0xffffffffu : (t < 0 ? 0u : ((2u << t) - 1u));
  }
}
// keep only bits c >= j (j <= 0: all, j > 127: none)
DEVI void set_bits_clear_below(uint32_t (&m)[4], int j) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int t = j - 32 * w;                  // lowest kept bit inside word w
    m[w] &= (t <= 0) ? 0xffffffffu : (t > 31 ? 0u : ~((1u << t) - 1u));
  }
}

// v[c] = fill where bit c of the (32 W)-bit mask m is clear.  A mask built from node runs is
// mostly whole 32-key words of ones or zeros (a run covers whole words, the causal edge cuts one
// word per row): those words take one test, only a mixed word is selected element by element.
template <int W, typename T>
DEVI void apply_mask_words(T (&v)[32 * W], const uint32_t (&m)[W], T fill) {
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const uint32_t b = m[w];
    if (b == 0xffffffffu) continue;
    if (b == 0u) {
#pragma unroll
      for (int c = 0; c < 32; ++c) v[32 * w + c] = fill;
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (!((b >> c) & 1u)) v[32 * w + c] = fill;
    }
  }
}

// fp32 RoPE inverse frequency theta^(-2c/d); shared by the forward rotation and the
// gradient's inverse rotation so that both use the same angles.
DEVI float rope_inv_freq(int c, int d, float theta) {
  return powf(theta, -static_cast<float>(2 * c) / static_cast<float>(d));
}

}  // namespace ta

// ------------------------------------------------------------------------------------------
// host-side helpers (defined in host.cu)
namespace ta {
int check_device();                                  // TREE_OK or TREE_ERR_ARCH / TREE_ERR_CUDA
int record_cuda(cudaError_t e);                      // TREE_OK or TREE_ERR_CUDA (message kept)
int make_tmap_bf16_3d(CUtensorMap* m, const void* base, int d, int heads, int rows);
int make_tmap_f32_2d(CUtensorMap* m, const void* base, int inner, int rows, int box_inner, int box_rows);
uint64_t wait_limit_ns();
int bwd_split_override();                            // 0: automatic
int fwd_split_override();                            // 0: automatic
int plan_ok(const tree_plan_t* p);
void record_timing_event(int i, cudaStream_t s);     // no-op unless events are registered
}  // namespace ta
