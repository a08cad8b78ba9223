// Grouped GEMM over the [E+B, H, H'] weight rows on 5th-generation tensor cores.
//
// "Moonshot AI 开源 MoonEP", contract paragraph: one weight tensor [E+B, H, H']
// per projection, rows [0,E) the home experts of every rank, rows [E, E+B) this
// rank's prefetch slots; cu_seqlens over the E+B rows selects the active rows.
// For rank u and group g the rows cu[u][g]..cu[u][g+1] of recv[u] are
// multiplied by W_home[g] (g < E) or by slot (u, g-E).
//
// Design (sm_103a):
//  * forward and input gradient: work tiles of 128 rows (k_ggemm_m128, one
//    CTA) or of 256 rows (k_ggemm_2sm on a CTA pair with the pair form of the
//    MMA when N is a multiple of 256, else k_ggemm_m256 on one CTA as two
//    128-row halves); every plan picks the height with the cost model of
//    gemm_cost.cuh and records it in the workspace.  Both heights are
//    launched; the one not chosen returns before touching anything.
//  * weight gradient: (group, 256 H rows, 256 H' columns) items on CTA pairs
//    (k_ggemm_dw_2sm) when H and H' are multiples of 256, else 128-row items
//    on one CTA (k_ggemm_dw); the accumulator is added into the fp32 gradient
//    with TMA reduce-adds.
//  * persistent CTAs (or CTA pairs), one per SM; the work list is the
//    planner's list of work tiles (or groups) of one group, times the column
//    tiles, claimed in order from a counter one item ahead.  Column tiles of
//    one row tile are adjacent in the order, so the items running together
//    share A rows and an expert's weights in L2.
//  * roles: warp 0 the TMA producer into a STAGES-deep shared-memory ring
//    (128-byte swizzled boxes); warp 1 TMEM allocation and the single-thread
//    tcgen05.mma issuer (bf16 x bf16 -> fp32 in TMEM, double-buffered
//    accumulators); warps 2..5 the epilogue: tcgen05.ld, bf16 rounding
//    (nearest even) and stores (TMA stores of 32-row slices in the pair
//    kernel, masked row stores where rows run past a group's end and in the
//    single-CTA kernels).
//  * every mbarrier wait is bounded by the global timer; on expiry the kernel
//    records MOONEP_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and
//    returns.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"

namespace moonep {

constexpr int kBK = 64;        // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;     // K of one tcgen05.mma for 16-bit inputs
constexpr int kGemmThreads = 192;
constexpr uint64_t kWaitNs = 4000000000ull;  // 4 s per barrier wait

constexpr int kQueueSlots = 16;  // work-item queue depth (kQueue below)

template <int BN, int STAGES>
struct GemmCfgM128 {  // one 128-row tile, double-buffered accumulator
  static constexpr int kABytes = kMmaM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kNumBars = 2 * STAGES + 5 + 2 * kQueueSlots;  // ring, TMEM, work-item queue
  static constexpr int kBarBytes = kNumBars * 8 + 16 + 4 * kQueueSlots;
  static constexpr int kSmem = STAGES * kStageBytes + 1024 + kBarBytes;
};

template <int BN, int STAGES>
struct GemmCfgM256 {  // two 128-row halves sharing each B stage
  static constexpr int kAHalf = kMmaM * kBK * 2;       // one 128-row A box
  static constexpr int kABytes = 2 * kAHalf;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;             // accumulators: cols [0,BN) and [BN,2BN)
  static constexpr int kBarBytes = (2 * STAGES + 5) * 8 + 16;
  static constexpr int kSmem = STAGES * kStageBytes + 1024 + kBarBytes;
};

// -- PTX wrappers -------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return (uint32_t)__cvta_generic_to_shared(ptr);
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity` to complete.  Gives up when the
// abort flag is raised by another role or after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)m) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* m, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"((uint64_t)m),
               "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_f32, uint32_t hi_f32) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(__uint_as_float(hi_f32)),
      "f"(__uint_as_float(lo_f32)));
  return out;
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format):
// start address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride
// byte offset >> 4 in 32-45, descriptor version 1 at bit 46, swizzle mode 2
// (128 B) in bits 61-63.  Tiles are 1024-byte aligned so the base offset is 0.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B
// bf16 (bits 7-9 = 1, 10-12 = 1), A K-major (bit 15 = 0), B N-major (bit 16 =
// 1), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn = false, bool b_mn = true) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Sizes of one grouped product: C[rows x N] = A[rows x K] . B[K x N], with B
// drawn from a weight tensor of wrows rows per expert.  Forward: K = H,
// N = H' (B = W, N-major).  Input gradient: K = H', N = H (B = W^T, which is
// W read K-major).
struct GemmShape {
  int K, N, wrows;
};

// B stage loads and descriptors for the two layouts of the weight operand.
template <int BN, bool BKM>
struct BOperand {
  // N-major: one box of BN/64 panels of 64(n) x 64(k), 8 KiB apart, from the
  // weights viewed as [H'/64][rows][64] (one TMA request instead of BN/64);
  // K-major: one box of 64(k) x BN(n) rows of 128 B.
  static __device__ __forceinline__ void load(uint32_t sb, const CUtensorMap* m, uint32_t bar,
                                              int n0, int k0, int wrow) {
    if (BKM) {
      tma_load_2d(sb, m, bar, k0, wrow + n0);
    } else {
      tma_load_3d(sb, m, bar, 0, wrow + k0, n0 / 64);
    }
  }
  static __device__ __forceinline__ uint64_t desc(uint32_t sb, int k) {
    return BKM ? sw128_desc(sb + k * (kUmmaK * 2), 16, 1024)
               : sw128_desc(sb + k * (kUmmaK * 128), 8192, 1024);
  }
};

// ---- pair (cta_group::2) PTX ----------------------------------------------
__device__ __forceinline__ uint32_t pair_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void pair_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// the shared::cluster address of this CTA's shared-memory word `a` in CTA `rank`
__device__ __forceinline__ uint32_t pair_map(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
// TMA load into this CTA's shared memory, completing bytes on an mbarrier that
// may sit in either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive once on the mbarrier at this offset in both CTAs of the pair when the
// MMAs issued so far by this thread have completed
__device__ __forceinline__ void umma_commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair_self(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Bounded wait with cluster-scope acquire, for barriers the other CTA of the
// pair arrives on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

// ---- work items of a CTA pair, claimed in order -------------------------------
// The pair's leader claims work items one at a time from a counter in global
// memory, one item ahead of the one it hands out (so the atomic's round trip
// overlaps an item's loads), and hands each to every role of both CTAs
// through a ring of kQueue shared-memory slots; -1 ends the sequence.  Claiming in order keeps the
// items that run at the same time contiguous in the work order (they share
// operand rows and weight panels in L2) and lets a pair that runs a little
// faster take more items: with a fixed stride the pairs drifted apart by the
// small, persistent speed differences between SMs (measured: about 1 % between
// the slowest and the fastest pairs, over two items of spread by the end of a
// pages-shaped forward GEMM).  The last pair to finish resets the counters for
// the next launch; the plan also zeroes them.
constexpr int kQueue = kQueueSlots;
constexpr int kQueueConsumers = 10;  // leader: MMA, 4 epilogue warps; peer: producer, 4 epilogue warps
constexpr int kQueueConsumersSolo = 5;  // a single CTA: MMA, 4 epilogue warps

struct PairQueue {
  uint32_t full0;   // this CTA's slot-0 "item written" barrier; slot s at full0 + 8 s
  uint32_t empty0;  // this CTA's slot-0 "item read" barrier (used in the leader)
  int32_t* items;   // this CTA's kQueue item slots
  __device__ uint32_t full(int s) const { return full0 + 8u * s; }
  __device__ uint32_t empty(int s) const { return empty0 + 8u * s; }
};

__device__ __forceinline__ void queue_init(const PairQueue& q, int consumers = kQueueConsumers) {
  for (int s = 0; s < kQueue; ++s) {
    mbar_init(q.full(s), 1);
    mbar_init(q.empty(s), consumers);
  }
}

// leader producer: the i-th claimed item t (or -1) into slot i % kQueue of both
// CTAs (of this CTA alone when `pair` is false: the same queue serves a
// kernel of single-CTA work items)
__device__ __forceinline__ bool queue_push(const PairQueue& q, int i, int t,
                                           volatile int* abort_flag, bool pair = true) {
  const int s = i % kQueue;
  if (!mbar_wait_cluster(q.empty(s), ((i / kQueue) & 1) ^ 1u, abort_flag)) return false;
  q.items[s] = t;
  if (pair) {
    const uint32_t remote = pair_map(smem_u32(q.items + s), 1);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(t) : "memory");
  }
  mbar_arrive(q.full(s));
  if (pair) mbar_arrive_remote(pair_map(q.full(s), 1));
  return true;
}

// a consumer thread (lane 0 of its role, or every lane of a warp with
// `arrive` on lane 0 only): the i-th item, then the slot released
__device__ __forceinline__ bool queue_take(const PairQueue& q, int i, bool leader, bool arrive,
                                           int& t, volatile int* abort_flag) {
  const int s = i % kQueue;
  if (!mbar_wait_cluster(q.full(s), (i / kQueue) & 1, abort_flag)) return false;
  t = *reinterpret_cast<volatile int32_t*>(q.items + s);
  if (arrive) {
    if (leader)
      asm volatile("mbarrier.arrive.release.cluster.shared::cta.b64 _, [%0];" ::"r"(q.empty(s))
                   : "memory");
    else
      mbar_arrive_remote(pair_map(q.empty(s), 0));
  }
  return true;
}

// a whole warp takes the i-th item; lane 0 releases the slot once every lane
// has read it
__device__ __forceinline__ bool queue_take_warp(const PairQueue& q, int i, bool leader, int& t,
                                                volatile int* abort_flag) {
  const int s = i % kQueue;
  if (!__all_sync(0xffffffffu, mbar_wait_cluster(q.full(s), (i / kQueue) & 1, abort_flag)))
    return false;
  t = *reinterpret_cast<volatile int32_t*>(q.items + s);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (leader)
      asm volatile("mbarrier.arrive.release.cluster.shared::cta.b64 _, [%0];" ::"r"(q.empty(s))
                   : "memory");
    else
      mbar_arrive_remote(pair_map(q.empty(s), 0));
  }
  return true;
}

// leader producer, once its pair has claimed past the end: the last pair of
// the launch resets the counters
__device__ __forceinline__ void queue_finish(int32_t* next, int32_t* finished, int pairs) {
  __threadfence();
  if (atomicAdd(finished, 1) == pairs - 1) {
    __threadfence();
    atomicExch(next, 0);
    atomicExch(finished, 0);
  }
}

// One 128-row tile per work item; the accumulator is double buffered so the
// epilogue of one tile overlaps the main loop of the next.
template <int BN, int STAGES, bool BKM>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_ggemm_m128(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_wh,
        const __grid_constant__ CUtensorMap tm_ws, Dims d, GemmShape sh, PlanPtrs p,
             uint16_t* __restrict__ y) {
  using Cfg = GemmCfgM128<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + STAGES * Cfg::kStageBytes);
  uint32_t* tmem_slot = (uint32_t*)(bars + Cfg::kNumBars);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);
  const PairQueue q{bar0 + 8u * (2 * STAGES + 5), bar0 + 8u * (2 * STAGES + 5 + kQueue),
                    (int32_t*)(tmem_slot + 2)};  // a queue of this CTA's own (no pair)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (plan_failed(p.status)) return;  // uniform: before any barrier or allocation
  if (p.counters[MOONEP_CNT_TILE_ROWS] != kMmaM) return;  // the plan chose 256-row tiles
  const int NT = sh.N / BN;
  const int total = p.counters[MOONEP_CNT_MTILES] * NT;
  const int KB = sh.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 4);
    }
    mbar_init(drain, 1);
    queue_init(q, kQueueConsumersSolo);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_wh);
    prefetch_tmap(&tm_ws);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      // items are claimed one ahead: the next claim travels while this item's
      // loads are issued
      int next = atomicAdd(p.sched + 4, 1);
      for (int i = 0; ok; ++i) {
        const int t = next >= total ? -1 : next;
        if (!queue_push(q, i, t, abort_flag, false)) { ok = false; break; }
        if (t >= 0) next = atomicAdd(p.sched + 4, 1);
        if (t < 0) break;
        const MTile mt = p.mtiles[t / NT];
        const int n0 = (t % NT) * BN;
        const CUtensorMap* wmap = mt.wsel >= 0 ? &tm_wh : &tm_ws;
        const int wrow = (mt.wsel >= 0 ? mt.wsel : (-1 - mt.wsel)) * sh.wrows;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          mbar_expect_tx(full(stage), Cfg::kStageBytes);
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          tma_load_2d(sa, &tm_a, full(stage), kb * kBK, mt.row0);
          BOperand<BN, BKM>::load(sa + Cfg::kABytes, wmap, full(stage), n0, kb * kBK, wrow);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      queue_finish(p.sched + 4, p.sched + 5, gridDim.x);
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        // wait (time-bounded) for the copies this thread started
        for (int i = 0; i < min(issued, STAGES); ++i) {
          if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
          mbar_wait(full(stage), phase, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kMmaM, BN, false, !BKM);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int t;
        if (!queue_take(q, i, true, true, t, abort_flag)) { ok = false; break; }
        if (t < 0) break;
        if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dtm = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sw128_desc(sa + k * (kUmmaK * 2), 16, 1024);
            const uint64_t bd = BOperand<BN, BKM>::desc(sb, k);
            umma_bf16(dtm, ad, bd, idesc, (kb | k) != 0);
          }
          umma_commit(empty(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        umma_commit(drain);  // completes once every MMA issued so far is done
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int qw = warp & 3;  // TMEM lanes 32qw..32qw+31 are this warp's rows
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = 0;; ++i) {
      int t;
      if (!queue_take_warp(q, i, true, t, abort_flag)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      if (t < 0) break;
      const MTile mt = p.mtiles[t / NT];
      const int n0 = (t % NT) * BN;
      const bool ok = mbar_wait(tfull(acc), acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const int row = qw * 32 + lane;
      const bool valid = row < mt.rows;
      uint16_t* yrow = y + (size_t)(mt.row0 + row) * sh.N + n0;
      const uint32_t tbase = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_x32(tbase + c * 32, r);
        tmem_ld_wait();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(yrow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o;
            o.x = pack_bf16x2(r[8 * v + 0], r[8 * v + 1]);
            o.y = pack_bf16x2(r[8 * v + 2], r[8 * v + 3]);
            o.z = pack_bf16x2(r[8 * v + 4], r[8 * v + 5]);
            o.w = pack_bf16x2(r[8 * v + 6], r[8 * v + 7]);
            dst[v] = o;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// 256-row work tiles on one CTA (N not a multiple of 256): two 128-row halves
// share every B stage, with two 128 x BN fp32 accumulators in TMEM (2*BN
// columns), so each byte of B fetched from L2 feeds twice the MMA work of a
// 128-row tile.  A tile whose group ends within its first half issues only the
// first half's MMAs.  Each accumulator is released as soon as it is drained,
// so the next tile's first-half MMAs overlap the drain of the second half.
template <int BN, int STAGES, bool BKM>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_ggemm_m256(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_wh,
             const __grid_constant__ CUtensorMap tm_ws, Dims d, GemmShape sh, PlanPtrs p,
             uint16_t* __restrict__ y) {
  using Cfg = GemmCfgM256<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + STAGES * Cfg::kStageBytes);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * STAGES + 5);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t tfull = bar0 + 8u * (2 * STAGES);
  auto tempty = [&](int h) { return bar0 + 8u * (2 * STAGES + 1 + h); };  // h = accumulator half
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (plan_failed(p.status)) return;  // uniform: before any barrier or allocation
  if (p.counters[MOONEP_CNT_TILE_ROWS] != 2 * kMmaM) return;  // the plan chose 128-row tiles
  const int NT = sh.N / BN;
  const int total = p.counters[MOONEP_CNT_MTILES] * NT;
  const int KB = sh.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty(0), 4);
    mbar_init(tempty(1), 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_wh);
    prefetch_tmap(&tm_ws);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const MTile mt = p.mtiles[t / NT];
        const int n0 = (t % NT) * BN;
        const bool two = mt.rows > kMmaM;
        const CUtensorMap* wmap = mt.wsel >= 0 ? &tm_wh : &tm_ws;
        const int wrow = (mt.wsel >= 0 ? mt.wsel : (-1 - mt.wsel)) * sh.wrows;
        const uint32_t bytes = Cfg::kAHalf * (two ? 2 : 1) + Cfg::kBBytes;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          mbar_expect_tx(full(stage), bytes);
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          tma_load_2d(sa, &tm_a, full(stage), kb * kBK, mt.row0);
          if (two) tma_load_2d(sa + Cfg::kAHalf, &tm_a, full(stage), kb * kBK, mt.row0 + kMmaM);
          BOperand<BN, BKM>::load(sa + Cfg::kABytes, wmap, full(stage), n0, kb * kBK, wrow);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        // wait (time-bounded) for the copies this thread started
        for (int i = 0; i < min(issued, STAGES); ++i) {
          if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
          mbar_wait(full(stage), phase, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kMmaM, BN, false, !BKM);
      int stage = 0;
      uint32_t phase = 0, item = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++item) {
        const bool two = p.mtiles[t / NT].rows > kMmaM;
        // accumulator h is free once the epilogue released it for the previous item
        if (!mbar_wait(tempty(0), (item & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sw128_desc(sa + k * (kUmmaK * 2), 16, 1024);
            const uint64_t bd = BOperand<BN, BKM>::desc(sb, k);
            umma_bf16(tmem_base, ad, bd, idesc, (kb | k) != 0);
          }
          if (two) {
            if (kb == 0) {
              if (!mbar_wait(tempty(1), (item & 1u) ^ 1u, abort_flag)) { ok = false; break; }
              tc_fence_after();
            }
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              const uint64_t ad = sw128_desc(sa + Cfg::kAHalf + k * (kUmmaK * 2), 16, 1024);
              const uint64_t bd = BOperand<BN, BKM>::desc(sb, k);
              umma_bf16(tmem_base + BN, ad, bd, idesc, (kb | k) != 0);
            }
          }
          umma_commit(empty(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(tfull);
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        umma_commit(drain);  // completes once every MMA issued so far is done
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;  // TMEM lanes 32q..32q+31 are this warp's rows
    uint32_t item = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++item) {
      const MTile mt = p.mtiles[t / NT];
      const int n0 = (t % NT) * BN;
      const bool ok = mbar_wait(tfull, item & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (h == 0 || mt.rows > kMmaM) {
          const int row = h * kMmaM + q * 32 + lane;
          const bool valid = row < mt.rows;
          uint16_t* yrow = y + (size_t)(mt.row0 + row) * sh.N + n0;
          const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * BN);
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_x32(tbase + c * 32, r);
            tmem_ld_wait();
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(yrow + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_bf16x2(r[8 * v + 0], r[8 * v + 1]);
                o.y = pack_bf16x2(r[8 * v + 2], r[8 * v + 3]);
                o.z = pack_bf16x2(r[8 * v + 4], r[8 * v + 5]);
                o.w = pack_bf16x2(r[8 * v + 6], r[8 * v + 7]);
                dst[v] = o;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(h));  // every item releases both halves
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// Tensor maps edited on the device: `map` (128 bytes in global memory, this
// thread's own copy) gets a new extent for dimension 1, and the edit is made
// visible to this thread's later TMA copies through the tensor-map proxy.
__device__ __forceinline__ void tmap_set_dim1(void* map, int extent) {
  asm volatile(
      "tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"((uint64_t)map),
      "r"(extent)
      : "memory");
}
__device__ __forceinline__ void tmap_publish(void* map) {
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"((uint64_t)map)
               : "memory");
}

// Ring depth of the pair kernel (32 KiB stages).  Measured with work items
// claimed in order, on one box: 6 stages 9.17-9.18 ms at the pages shape and
// 5.44-5.46 ms at the K3 shape, against 9.23-9.30 and 5.53-5.54 ms with 5.
// (With a fixed stride per pair the sixth stage had been slower, 9.2 against
// 9.0 ms: the pairs drifted further apart and panels were evicted before
// their last reader, 38-41 GB of DRAM reads per launch against 29.)
constexpr int kPairStages = 6;

template <int STAGES>
struct GemmCfgPair {  // per CTA: its 128 rows of A and 128 of the 256 columns of B
  static constexpr int kABytes = kMmaM * kBK * 2;
  static constexpr int kBBytes = 128 * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 512;  // two 128-lane x 256-column fp32 accumulators
  // output staging: per epilogue warp two 32-row x 64-column bf16 buffers
  // (128-byte rows, 128-byte swizzle), the sources of its TMA stores
  static constexpr int kOutWarpBytes = 2 * 4096;
  static constexpr int kOutBytes = 4 * kOutWarpBytes;
  static constexpr int kNumBars = 2 * STAGES + 5 + 2 * kQueue;
  static constexpr int kBarBytes = kNumBars * 8 + 16 + 4 * kQueue;
  static constexpr int kSmem = STAGES * kStageBytes + kOutBytes + 1024 + kBarBytes;
};

// 256 x 256 work tiles on a CTA pair with the pair form of the MMA
// (tcgen05 cta_group::2, M = 256): CTA c of a two-CTA cluster holds rows
// 128c..128c+127 of the tile's A and columns 128c..128c+127 of its B panel;
// one MMA instruction computes the whole 256 x 256 x 16 product, each SM's
// tensor core producing its 128 rows from its own A and both halves of B.
// Per K block each SM so loads 32 KiB for 128 x 256 x 64 of MMA work, where
// the single-CTA 128-row kernel loads 48 KiB for the same work, and the
// smaller stage buys a deeper ring.
// CTA 0 (the leader) issues the MMAs and owns the full, tempty and drain
// barriers; both CTAs' loads complete on the leader's full barrier; each MMA
// commit arrives on the empty (or tfull) barrier of both CTAs; each CTA drains
// its own 128 accumulator rows and releases them on the leader's tempty.
// Items are the 256-row tiles of the plan times N/256 column tiles, claimed in
// order by the pair (PairQueue).  A group's last tile has rows past the
// group's end; they are loaded as zeros, so the MMAs on them multiply zeros
// (their results are never stored): a tile of at most 128 rows leaves the
// second CTA's rows unused and that CTA's A box starts past the end of recv,
// and a CTA whose rows run past the group's end loads them through its own
// copy of the A tensor map with the row extent cut at the group's end (a ring
// of kTmapSlots copies in the plan workspace, as the weight gradient uses).
// BKM = false: the
// forward product (B = W, N-major, two 64-column panels per CTA from one 3D
// box); BKM = true: the input gradient (B = W^T, i.e. W read K-major, 128
// weight rows per CTA).
template <int STAGES, bool BKM>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
k_ggemm_2sm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_wh,
            const __grid_constant__ CUtensorMap tm_ws, const __grid_constant__ CUtensorMap tm_y,
            Dims d, GemmShape sh, PlanPtrs p, uint16_t* __restrict__ y) {
  using Cfg = GemmCfgPair<STAGES>;
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* out_stage = smem + STAGES * Cfg::kStageBytes;  // 1024-aligned
  uint64_t* bars = (uint64_t*)(out_stage + Cfg::kOutBytes);
  uint32_t* tmem_slot = (uint32_t*)(bars + Cfg::kNumBars);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);
  const PairQueue q{bar0 + 8u * (2 * STAGES + 5), bar0 + 8u * (2 * STAGES + 5 + kQueue),
                    (int32_t*)(tmem_slot + 2)};
  constexpr uint64_t kDrainNs = 200000000ull;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = pair_rank();
  const bool leader = crank == 0;
  const int ncl = gridDim.x >> 1;
  if (plan_failed(p.status)) return;  // uniform over the pair: before any barrier
  if (p.counters[MOONEP_CNT_TILE_ROWS] != 2 * kMmaM) return;
  const int NT = sh.N / BN;
  const int total = p.counters[MOONEP_CNT_MTILES] * NT;
  const int KB = sh.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 8);  // four epilogue warps in each CTA
    }
    mbar_init(drain, 1);
    queue_init(q);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_wh);
    prefetch_tmap(&tm_ws);
    prefetch_tmap(&tm_y);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pair_sync();  // the peer's barriers are initialised before anything reaches them
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      // this CTA's ring of A tensor-map copies (the first map of each slot)
      uint4* maps = reinterpret_cast<uint4*>(p.tmaps) + (size_t)blockIdx.x * kTmapSlots * 16;
      {
        const uint4* sa0 = reinterpret_cast<const uint4*>(&tm_a);
        for (int i = 0; i < kTmapSlots; ++i)
          for (int j = 0; j < 8; ++j) maps[i * 16 + j] = sa0[j];
      }
      int stage = 0, issued = 0, slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      // the leader claims one item ahead: the claim of the next item travels
      // while this one's loads are issued
      int next = leader ? atomicAdd(p.sched, 1) : 0;
      for (int i = 0; ok; ++i) {
        int t;
        if (leader) {  // hand the claimed item to the pair, claim the following one
          t = next >= total ? -1 : next;
          if (!queue_push(q, i, t, abort_flag)) { ok = false; break; }
          if (t >= 0) next = atomicAdd(p.sched, 1);
        } else if (!queue_take(q, i, false, true, t, abort_flag)) {
          ok = false;
          break;
        }
        if (t < 0) break;
        const MTile mt = p.mtiles[t / NT];
        const int n0 = (t % NT) * BN + (int)crank * 128;
        const CUtensorMap* wmap = mt.wsel >= 0 ? &tm_wh : &tm_ws;
        const int wrow = (mt.wsel >= 0 ? mt.wsel : (-1 - mt.wsel)) * sh.wrows;
        // the second CTA's rows of a tile of at most 128 rows are unused: its
        // box starts past the last row of A, so TMA fills it with zeros and
        // reads nothing
        const int row0 = (crank == 0 || mt.rows > kMmaM) ? mt.row0 + (int)crank * kMmaM : d.R * d.C;
        const CUtensorMap* amap = &tm_a;
        if (row0 < d.R * d.C && mt.rows < (int)(crank + 1) * kMmaM) {
          // this CTA's rows run past the group's end: rows from there on read as zeros
          uint4* m = maps + slot * 16;
          tmap_set_dim1(m, mt.row0 + mt.rows);
          tmap_publish(m);
          amap = reinterpret_cast<const CUtensorMap*>(m);
          if (++slot == kTmapSlots) slot = 0;
        }
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t fb = pair_map(full(stage), 0);
          if (leader) mbar_expect_tx(full(stage), 2 * Cfg::kStageBytes);
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          tma_load_2d_pair(sa, amap, fb, kb * kBK, row0);
          if (BKM)  // 128 weight rows (this CTA's n), 64 k each
            tma_load_2d_pair(sa + Cfg::kABytes, wmap, fb, kb * kBK, wrow + n0);
          else      // two 64-column panels of 64 k-rows
            tma_load_3d_pair(sa + Cfg::kABytes, wmap, fb, 0, wrow + kb * kBK, n0 / 64);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader) queue_finish(p.sched, p.sched + 1, ncl);
      if (ok) {
        for (int i = 0; i < STAGES; ++i) {  // every fill released: no commit still in flight
          if (!mbar_wait(empty(stage), phase ^ 1u, nullptr)) { ok = false; break; }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) set_error(p.status, MOONEP_ERR_TIMEOUT);
      } else {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        if (leader) {
          for (int i = 0; i < min(issued, STAGES); ++i) {
            if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
            mbar_wait(full(stage), phase, nullptr, kDrainNs);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader only) ----------------
    if (leader && lane == 0) {
      constexpr uint32_t idesc = make_idesc(2 * kMmaM, BN, false, !BKM);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int t;
        if (!queue_take(q, i, true, true, t, abort_flag)) { ok = false; break; }
        if (t < 0) break;
        if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dtm = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sw128_desc(sa + k * (kUmmaK * 2), 16, 1024);
            const uint64_t bd = BKM ? sw128_desc(sb + k * (kUmmaK * 2), 16, 1024)
                                    : sw128_desc(sb + k * (kUmmaK * 128), 8192, 1024);
            umma_bf16_pair(dtm, ad, bd, idesc, (kb | k) != 0);
          }
          umma_commit_pair_both(empty(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair_both(tfull(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        umma_commit_pair_self(drain);
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5, both CTAs) ----------------
    const int qw = warp & 3;
    int acc = 0, nstore = 0;
    uint32_t acc_phase = 0;
    for (int i = 0;; ++i) {
      int t;
      if (!queue_take_warp(q, i, leader, t, abort_flag)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      if (t < 0) break;
      const MTile mt = p.mtiles[t / NT];
      const int n0 = (t % NT) * BN;
      const bool ok = mbar_wait(tfull(acc), acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const int wrow0 = (int)crank * kMmaM + qw * 32;  // this warp's first row of the tile
      const uint32_t tbase = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(acc * BN);
      if (wrow0 + 32 <= mt.rows) {
        // all 32 rows inside the group: bf16 rows staged in shared memory
        // (128-byte swizzle, so the lanes of a store phase hit distinct bank
        // groups) and written by one TMA store per 64 columns
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c, ++nstore) {
          uint32_t lo[32], hi[32];
          tmem_ld_x32(tbase + c * 64, lo);
          tmem_ld_x32(tbase + c * 64 + 32, hi);
          tmem_ld_wait();
          uint8_t* buf = out_stage + qw * Cfg::kOutWarpBytes + (nstore & 1) * 4096;
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          __syncwarp();
          uint4* rowp = reinterpret_cast<uint4*>(buf + lane * 128);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            rowp[v ^ (lane & 7)] =
                make_uint4(pack_bf16x2(lo[8 * v + 0], lo[8 * v + 1]), pack_bf16x2(lo[8 * v + 2], lo[8 * v + 3]),
                           pack_bf16x2(lo[8 * v + 4], lo[8 * v + 5]), pack_bf16x2(lo[8 * v + 6], lo[8 * v + 7]));
            rowp[(4 + v) ^ (lane & 7)] =
                make_uint4(pack_bf16x2(hi[8 * v + 0], hi[8 * v + 1]), pack_bf16x2(hi[8 * v + 2], hi[8 * v + 3]),
                           pack_bf16x2(hi[8 * v + 4], hi[8 * v + 5]), pack_bf16x2(hi[8 * v + 6], hi[8 * v + 7]));
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            asm volatile(
                "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                    (uint64_t)&tm_y),
                "r"(n0 + c * 64), "r"(mt.row0 + wrow0), "r"(smem_u32(buf))
                : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      } else {
        // rows past the group's end belong to the next group: each lane
        // stores its own row if it is inside the group
        const int row = wrow0 + lane;
        const bool valid = row < mt.rows;
        uint16_t* yrow = y + (size_t)(mt.row0 + row) * sh.N + n0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_x32(tbase + c * 32, r);
          tmem_ld_wait();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              o.x = pack_bf16x2(r[8 * v + 0], r[8 * v + 1]);
              o.y = pack_bf16x2(r[8 * v + 2], r[8 * v + 3]);
              o.z = pack_bf16x2(r[8 * v + 4], r[8 * v + 5]);
              o.w = pack_bf16x2(r[8 * v + 6], r[8 * v + 7]);
              dst[v] = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(pair_map(tempty(acc), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // this warp's stores
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  pair_sync();  // both CTAs done with TMEM and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

// Weight gradient of the grouped GEMM: for every non-empty (rank u, weight
// row g) group with rows a0..a1 of the receive buffer,
//   G(u,g) += X[a0:a1]^T . dY[a0:a1]        ([H x H'], fp32),
// where G(u,g) is g_home[g] for a home group and slot (u, g-E) of g_slot for a
// slot group ("Moonshot AI 开源 MoonEP", contract paragraph: the redundant
// experts' gradients go to the [R, B, H, H'] reduce buffers that reduce_grad
// folds into the home rows).  Work items are (group, 128-row tile of H, BN
// column tile of H'), H tiles fastest (3.5 % faster than H' tiles fastest at
// the K3 shape, equal at the pages shape), so the CTAs running together read
// the same group's rows from L2.  Both operands are read N-major straight from
// the row-major buffers, each stage by two 3D boxes: A = X^T (2 panels of
// 64(h) x 64(row)), B = dY (BN/64 panels of 64(n) x 64(row)).  The reduction
// runs over the group's rows in 64-row blocks; in the last block the rows past
// the group's end are zeroed in shared memory before the MMAs.  Accumulators
// are double buffered in TMEM.  The four epilogue warps stage a 128 x 64 fp32
// chunk together in shared memory and one thread adds it into G with a TMA
// reduce-add, so the read-modify-write happens in L2.  Every G element gets
// one add per launch, always a cold line: for groups long enough to hide it,
// the producer asks L2 to prefetch the item's G tile when the item starts, so
// the reduce-adds at its end find the lines resident.
// The weight gradient prefetches a work item's G tile into L2 only when the
// item reduces over at least this many 64-row blocks (measured: shorter items
// leave too little time for the prefetch and only add DRAM traffic).
constexpr int kDwPrefetchMinBlocks = 16;

// Permutes the eight 16-byte vectors held in r (four words each) so that slot j
// holds the vector that was in slot j ^ m (m < 8): three conditional swap stages,
// one per bit of m, with register indices fixed at compile time.
__device__ __forceinline__ void xor_vectors8(uint32_t (&r)[32], int m) {
#pragma unroll
  for (int b = 1; b < 8; b <<= 1) {
    const bool s = (m & b) != 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j & b) continue;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x = r[4 * j + w], y = r[4 * (j ^ b) + w];
        r[4 * j + w] = s ? y : x;
        r[4 * (j ^ b) + w] = s ? x : y;
      }
    }
  }
}

template <int BN, int STAGES>
struct GemmCfgDW {
  static constexpr int kABytes = kMmaM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kOutBytes = 32768;  // 128 rows x 64 fp32, 256-byte rows, no swizzle
  static constexpr int kBarBytes = (2 * STAGES + 5) * 8 + 16;
  static constexpr int kSmem = STAGES * kStageBytes + kOutBytes + 1024 + kBarBytes;
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_ggemm_dw(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
           const __grid_constant__ CUtensorMap tm_gh, const __grid_constant__ CUtensorMap tm_gs,
           const __grid_constant__ CUtensorMap tm_ghp, const __grid_constant__ CUtensorMap tm_gsp,
           Dims d, PlanPtrs p) {
  using Cfg = GemmCfgDW<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* out_stage = smem + STAGES * Cfg::kStageBytes;  // 1024-aligned
  uint64_t* bars = (uint64_t*)(out_stage + Cfg::kOutBytes);
  uint32_t* tmem_slot = (uint32_t*)(bars + 2 * STAGES + 5);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (plan_failed(p.status)) return;  // uniform: before any barrier or allocation
  const int MT = d.H / kMmaM, NT = d.Hp / BN;
  const int per_group = MT * NT;
  const int total = p.counters[MOONEP_CNT_GROUPS] * per_group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_dy);
    prefetch_tmap(&tm_gh);
    prefetch_tmap(&tm_gs);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const MTile grp = p.groups[t / per_group];
        const int m0 = ((t % per_group) % MT) * kMmaM;
        const int n0 = ((t % per_group) / MT) * BN;
        const int KB = (grp.rows + kBK - 1) / kBK;
        if (KB >= kDwPrefetchMinBlocks)
          tma_prefetch_2d(grp.wsel >= 0 ? &tm_ghp : &tm_gsp, n0,
                          (grp.wsel >= 0 ? grp.wsel : (-1 - grp.wsel)) * d.H + m0);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          mbar_expect_tx(full(stage), Cfg::kStageBytes);
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          const int r0 = grp.row0 + kb * kBK;
          tma_load_3d(sa, &tm_x, full(stage), 0, r0, m0 / 64);
          tma_load_3d(sa + Cfg::kABytes, &tm_dy, full(stage), 0, r0, n0 / 64);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        for (int i = 0; i < min(issued, STAGES); ++i) {
          if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
          mbar_wait(full(stage), phase, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (lane 0) with partial-block zeroing (all lanes) ----
    constexpr uint32_t idesc = make_idesc(kMmaM, BN, true, true);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const MTile grp = p.groups[t / per_group];
      const int KB = (grp.rows + kBK - 1) / kBK;
      ok = __all_sync(0xffffffffu, mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t dtm = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < KB; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(full(stage), phase, abort_flag));
        if (!ok) break;
        uint8_t* st_base = smem + stage * Cfg::kStageBytes;
        const int valid = grp.rows - kb * kBK;
        if (valid < kBK) {  // rows past the group's end belong to another group
          constexpr int kBoxes = 2 + BN / 64;
          const int per_box = (kBK - valid) * 8;  // uint4 per box
          for (int i = lane; i < kBoxes * per_box; i += 32) {
            const int box = i / per_box, j = i % per_box;
            uint4* z = reinterpret_cast<uint4*>(st_base + box * 8192 + valid * 128) + j;
            *z = make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sa = smem_u32(st_base);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sw128_desc(sa + k * (kUmmaK * 128), 8192, 1024);
            const uint64_t bd = sw128_desc(sb + k * (kUmmaK * 128), 8192, 1024);
            umma_bf16(dtm, ad, bd, idesc, (kb | k) != 0);
          }
          umma_commit(empty(stage));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(tfull(acc));
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_error(p.status, MOONEP_ERR_TIMEOUT);
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else {
    // ---------------- epilogue (warps 2..5): G += accumulator ----------------
    // Each warp owns 32 rows of the tile.  The tile is drained in 128 x 64 fp32
    // chunks: each row's 64 columns go from TMEM into a plain row-major staging
    // buffer (256-byte rows) and one thread adds the chunk into G with a TMA
    // reduce (the read-modify-write happens in L2); the buffer is reused once
    // the reduce that read it is done.
    const int q = warp & 3;
    const bool issuer = (warp == 2 && lane == 0);
    auto epi_bar = []() { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    auto epi_all = [](bool pred) {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
          "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
          : "=r"(r)
          : "r"((uint32_t)pred)
          : "memory");
      return r != 0;
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const MTile grp = p.groups[t / per_group];
      const int m0 = ((t % per_group) % MT) * kMmaM;
      const int n0 = ((t % per_group) / MT) * BN;
      const bool okw = mbar_wait(tfull(acc), acc_phase, abort_flag);
      if (!epi_all(okw)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const CUtensorMap* gmap = grp.wsel >= 0 ? &tm_gh : &tm_gs;
      const int grow = (grp.wsel >= 0 ? grp.wsel : (-1 - grp.wsel)) * d.H + m0;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const int rr = q * 32 + lane;
      const int m = rr & 7;
      uint4* row = reinterpret_cast<uint4*>(out_stage + rr * 256);
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t lo[32], hi[32];
        tmem_ld_x32(tbase + c * 64, lo);
        tmem_ld_x32(tbase + c * 64 + 32, hi);
        tmem_ld_wait();
        xor_vectors8(lo, m);
        xor_vectors8(hi, m);
        if (issuer) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        epi_bar();
        // vector order j ^ (row & 7): the eight lanes of a store phase hit eight
        // different bank groups
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          row[j ^ m] = make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
          row[8 + (j ^ m)] = make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epi_bar();
        if (issuer) {
          asm volatile(
              "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
              " [%0, {%1, %2}], [%3];" ::"l"((uint64_t)gmap),
              "r"(n0 + c * 64), "r"(grow), "r"(smem_u32(out_stage))
              : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (issuer) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// Weight gradient on CTA pairs (tcgen05 cta_group::2, M = 256 rows of H,
// N = 256 columns of H').  Work items are (group, 256-row tile of H,
// 256-column tile of H'), H tiles fastest.  CTA c of the pair holds H rows
// 128c.. of the tile's A = X^T and H' columns 128c.. of its B = dY, each as
// two 64-wide panels of 64 group rows per stage: 32 KiB per SM per stage for
// the MMA work the single-CTA kernel feeds with 48 KiB, so the ring is six
// stages deep in the same shared memory and a third fewer operand bytes cross
// from L2.  Each CTA drains its own 128 x 256 accumulator into G by TMA
// reduce-adds, as the single-CTA kernel does.
// The 64-row block that runs past a group's end is loaded through copies of
// the recv and dY tensor maps whose row extent ends at the group's end, so TMA
// fills the rows past it with zeros: every block of every item then completes
// on the leader's barrier and no block needs a shared-memory fix-up.  Each CTA
// keeps a ring of kTmapSlots such copies in the plan workspace; a copy is
// rewritten only after the load that used it has completed (the ring is deeper
// than the stage ring, and a stage is refilled only once its previous load
// has been consumed).
constexpr int kDwPairStages = 6;

template <int STAGES>
struct GemmCfgDWPair {
  static constexpr int kABytes = kMmaM * kBK * 2;  // 128 H rows x 64 group rows
  static constexpr int kBBytes = 128 * kBK * 2;    // 128 H' columns x 64 group rows
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 512;            // two 128-lane x 256-column fp32 accumulators
  static constexpr int kOutBytes = 32768;          // 128 rows x 64 fp32, 256-byte rows, no swizzle
  static constexpr int kNumBars = 2 * STAGES + 5 + 2 * kQueue;
  static constexpr int kBarBytes = kNumBars * 8 + 16 + 4 * kQueue;
  static constexpr int kSmem = STAGES * kStageBytes + kOutBytes + 1024 + kBarBytes;
};
static_assert(kTmapSlots > kDwPairStages, "a tensor-map copy must outlive the loads in flight");

template <int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
k_ggemm_dw_2sm(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
               const __grid_constant__ CUtensorMap tm_gh, const __grid_constant__ CUtensorMap tm_gs,
               Dims d, PlanPtrs p) {
  using Cfg = GemmCfgDWPair<STAGES>;
  constexpr int BN = 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* out_stage = smem + STAGES * Cfg::kStageBytes;  // 1024-aligned
  uint64_t* bars = (uint64_t*)(out_stage + Cfg::kOutBytes);
  uint32_t* tmem_slot = (uint32_t*)(bars + Cfg::kNumBars);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);
  const PairQueue q{bar0 + 8u * (2 * STAGES + 5), bar0 + 8u * (2 * STAGES + 5 + kQueue),
                    (int32_t*)(tmem_slot + 2)};
  constexpr uint64_t kDrainNs = 200000000ull;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = pair_rank();
  const bool leader = crank == 0;
  const int ncl = gridDim.x >> 1;
  if (plan_failed(p.status)) return;  // uniform over the pair: before any barrier
  const int MT = d.H / (2 * kMmaM), NT = d.Hp / BN;
  const int per_group = MT * NT;
  const int total = p.counters[MOONEP_CNT_GROUPS] * per_group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), 8);  // four epilogue warps in each CTA
    }
    mbar_init(drain, 1);
    queue_init(q);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_dy);
    prefetch_tmap(&tm_gh);
    prefetch_tmap(&tm_gs);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pair_sync();  // the peer's barriers are initialised before anything reaches them
  const uint32_t tmem_base = *tmem_slot;

  // work item t: its group, first H row and first H' column (every role of
  // both CTAs walks the same sequence)
  auto item = [&](int t, MTile& grp, int& m0, int& n0) {
    grp = p.groups[t / per_group];
    const int r = t % per_group;
    m0 = (r % MT) * (2 * kMmaM);
    n0 = (r / MT) * BN;
  };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      // this CTA's ring of tensor-map copies (recv, dY) for the blocks that
      // run past a group's end
      uint4* maps = reinterpret_cast<uint4*>(p.tmaps) + (size_t)blockIdx.x * kTmapSlots * 16;
      {
        const uint4* sx = reinterpret_cast<const uint4*>(&tm_x);
        const uint4* sy = reinterpret_cast<const uint4*>(&tm_dy);
        for (int i = 0; i < kTmapSlots; ++i)
          for (int j = 0; j < 8; ++j) {
            maps[i * 16 + j] = sx[j];
            maps[i * 16 + 8 + j] = sy[j];
          }
      }
      int stage = 0, issued = 0, slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      // the leader claims one item ahead: the claim of the next item travels
      // while this one's loads are issued
      int next = leader ? atomicAdd(p.sched + 2, 1) : 0;
      for (int i = 0; ok; ++i) {
        int t;
        if (leader) {  // hand the claimed item to the pair, claim the following one
          t = next >= total ? -1 : next;
          if (!queue_push(q, i, t, abort_flag)) { ok = false; break; }
          if (t >= 0) next = atomicAdd(p.sched + 2, 1);
        } else if (!queue_take(q, i, false, true, t, abort_flag)) {
          ok = false;
          break;
        }
        if (t < 0) break;
        MTile grp;
        int m0, n0;
        item(t, grp, m0, n0);
        const int KB = (grp.rows + kBK - 1) / kBK;
        const int hrow = m0 + (int)crank * kMmaM;  // this CTA's H rows: columns of recv
        const int ncol = n0 + (int)crank * 128;    // this CTA's H' columns of dY
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          const int r0 = grp.row0 + kb * kBK;
          const CUtensorMap* mx = &tm_x;
          const CUtensorMap* my = &tm_dy;
          if (grp.rows - kb * kBK < kBK) {
            // the group's partial last block: rows from the group's end on read as zeros
            uint4* m = maps + slot * 16;
            tmap_set_dim1(m, grp.row0 + grp.rows);
            tmap_set_dim1(m + 8, grp.row0 + grp.rows);
            tmap_publish(m);
            tmap_publish(m + 8);
            mx = reinterpret_cast<const CUtensorMap*>(m);
            my = reinterpret_cast<const CUtensorMap*>(m + 8);
            if (++slot == kTmapSlots) slot = 0;
          }
          // both CTAs' loads complete on the leader's full barrier
          const uint32_t fb = pair_map(full(stage), 0);
          if (leader) mbar_expect_tx(full(stage), 2 * Cfg::kStageBytes);
          tma_load_3d_pair(sa, mx, fb, 0, r0, hrow / 64);
          tma_load_3d_pair(sa + Cfg::kABytes, my, fb, 0, r0, ncol / 64);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (leader) queue_finish(p.sched + 2, p.sched + 3, ncl);
      if (ok) {
        for (int i = 0; i < STAGES; ++i) {  // every fill released: no commit still in flight
          if (!mbar_wait(empty(stage), phase ^ 1u, nullptr)) { ok = false; break; }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) set_error(p.status, MOONEP_ERR_TIMEOUT);
      } else {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        if (leader) {  // both CTAs' copies complete on the leader's barriers
          for (int i = 0; i < min(issued, STAGES); ++i) {
            if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
            mbar_wait(full(stage), phase, nullptr, kDrainNs);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader only) ----------------
    if (leader && lane == 0) {
      constexpr uint32_t idesc = make_idesc(2 * kMmaM, BN, true, true);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int t;
        if (!queue_take(q, i, true, true, t, abort_flag)) { ok = false; break; }
        if (t < 0) break;
        const int KB = (p.groups[t / per_group].rows + kBK - 1) / kBK;
        if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dtm = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(full(stage), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sw128_desc(sa + k * (kUmmaK * 128), 8192, 1024);
            const uint64_t bd = sw128_desc(sb + k * (kUmmaK * 128), 8192, 1024);
            umma_bf16_pair(dtm, ad, bd, idesc, (kb | k) != 0);
          }
          umma_commit_pair_both(empty(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair_both(tfull(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        *abort_flag = 1;
        set_error(p.status, MOONEP_ERR_TIMEOUT);
        umma_commit_pair_self(drain);  // completes once every MMA issued so far is done
        mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5, both CTAs): G += accumulator ----------------
    const int qw = warp & 3;
    const bool issuer = (warp == 2 && lane == 0);
    auto epi_bar = []() { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    auto epi_all = [](bool pred) {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
          "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
          : "=r"(r)
          : "r"((uint32_t)pred)
          : "memory");
      return r != 0;
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = 0;; ++i) {
      int t;
      if (!queue_take_warp(q, i, leader, t, abort_flag)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      if (t < 0) break;
      MTile grp;
      int m0, n0;
      item(t, grp, m0, n0);
      const bool okw = mbar_wait(tfull(acc), acc_phase, abort_flag);
      if (!epi_all(okw)) {
        if (lane == 0) {
          *abort_flag = 1;
          set_error(p.status, MOONEP_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const CUtensorMap* gmap = grp.wsel >= 0 ? &tm_gh : &tm_gs;
      const int grow = (grp.wsel >= 0 ? grp.wsel : (-1 - grp.wsel)) * d.H + m0 + (int)crank * kMmaM;
      const uint32_t tbase = tmem_base + ((uint32_t)(qw * 32) << 16) + (uint32_t)(acc * BN);
      const int rr = qw * 32 + lane;
      const int m = rr & 7;
      uint4* row = reinterpret_cast<uint4*>(out_stage + rr * 256);
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c) {
        // this row's 64 columns: 16 vectors of 16 bytes, read from TMEM while the
        // previous chunk's reduce-add may still be reading the buffer
        uint32_t lo[32], hi[32];
        tmem_ld_x32(tbase + c * 64, lo);
        tmem_ld_x32(tbase + c * 64 + 32, hi);
        tmem_ld_wait();
        xor_vectors8(lo, m);
        xor_vectors8(hi, m);
        if (issuer) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        epi_bar();
        // the buffer is plain row-major (256-byte rows); each lane writes its
        // vectors in the order j ^ (row & 7), so the eight lanes of a store phase
        // hit eight different bank groups
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          row[j ^ m] = make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
          row[8 + (j ^ m)] = make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        epi_bar();
        if (issuer) {
          asm volatile(
              "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
              " [%0, {%1, %2}], [%3];" ::"l"((uint64_t)gmap),
              "r"(n0 + c * 64), "r"(grow), "r"(smem_u32(out_stage))
              : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(pair_map(tempty(acc), 0));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (issuer) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  pair_sync();  // both CTAs done with TMEM and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// ever arrives on, with the same helper the GEMM pipeline uses, and must give up
// after limit_ns, record MOONEP_ERR_TIMEOUT and return.
__global__ void k_wait_selftest(int32_t* status, uint64_t limit_ns, int32_t* elapsed_us) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    if (!mbar_wait(smem_u32(&bar), 0, nullptr, limit_ns)) set_error(status, MOONEP_ERR_TIMEOUT);
    *elapsed_us = (int32_t)((global_ns() - t0) / 1000);
  }
}

cudaError_t launch_wait_selftest(int32_t* status, uint32_t limit_us, int32_t* elapsed_us,
                                 cudaStream_t st, int* launches) {
  k_wait_selftest<<<1, 32, 0, st>>>(status, (uint64_t)limit_us * 1000ull, elapsed_us);
  *launches += 1;
  return cudaGetLastError();
}

// -- host side ------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* sym = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &sym, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)sym;
  }
  return fn;
}

// 2D bf16 tensor [outer][inner], box [box_outer][64], 128-byte swizzle.
static bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_outer) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t gdim[2] = {inner, outer};
  cuuint64_t gstride[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major bf16 matrix [rows][inner] viewed as [inner/64][rows][64]: one
// box is nchunk 128-byte-swizzled panels of 64 rows x 64 columns, 8 KiB apart
// in shared memory, the same layout as nchunk 2D boxes of 64 x 64.
static bool encode_panels_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                             uint32_t nchunk) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t gdim[3] = {64, rows, inner / 64};
  cuuint64_t gstride[2] = {inner * 2, 128};
  cuuint32_t box[3] = {64, 64, nchunk};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 tensor [outer][inner] with a box of 128 rows x box_inner, no swizzle
// (L2 prefetch of a weight-gradient tile; with 64 columns, the reduce-add
// target of the weight-gradient kernels).
static bool encode_2d_f32_tile(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                               uint32_t box_inner) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t gdim[2] = {inner, outer};
  cuuint64_t gstride[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Cfg, typename KernelT, typename... Args>
static cudaError_t launch_cfg(KernelT kernel, bool& attr_set, int grid, cudaStream_t st,
                              Args... args) {
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kernel<<<grid, kGemmThreads, Cfg::kSmem, st>>>(args...);
  return cudaGetLastError();
}

template <int BN, int S128, int S256, bool BKM>
static cudaError_t launch_bn(const Dims& d, GemmShape sh, const PlanPtrs& p, const CUtensorMap& a,
                             const CUtensorMap& wh, const CUtensorMap& ws, uint16_t* y, int grid,
                             cudaStream_t st, int* launches) {
  // With the height left to the plan both variants are launched; the one the
  // plan did not choose returns at once (the choice is only on the device).
  static bool set128 = false, set256 = false;
  int n = 0;
  if (d.tile_m != 2 * kMmaM) {
    const cudaError_t e = launch_cfg<GemmCfgM128<BN, S128>>(k_ggemm_m128<BN, S128, BKM>, set128,
                                                            grid, st, a, wh, ws, d, sh, p, y);
    if (e != cudaSuccess) return e;
    ++n;
  }
  if (d.tile_m != kMmaM) {
    const cudaError_t e = launch_cfg<GemmCfgM256<BN, S256>>(k_ggemm_m256<BN, S256, BKM>, set256,
                                                            grid, st, a, wh, ws, d, sh, p, y);
    if (e != cudaSuccess) return e;
    ++n;
  }
  *launches += n;
  return cudaSuccess;
}

static int sm_count_gemm() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

static int pick_bn(int n) { return (n % 256 == 0) ? 256 : (n % 128 == 0 ? 128 : 64); }

static bool set_fwd128 = false, set_dx128 = false;

// The CTA-pair kernel on two CTAs per co-resident cluster.
template <bool BKM>
static cudaError_t launch_pair_gemm(const Dims& d, GemmShape sh, const PlanPtrs& p,
                                    const CUtensorMap& a, const CUtensorMap& wh,
                                    const CUtensorMap& ws, uint16_t* y, cudaStream_t st) {
  using Cfg = GemmCfgPair<kPairStages>;
  CUtensorMap ty;  // the output as TMA store target, 32-row boxes of 64 columns
  if (!encode_2d(&ty, y, (uint64_t)sh.N, (uint64_t)d.R * d.C, 32)) return cudaErrorInvalidValue;
  static int grid = 0;
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_ggemm_2sm<kPairStages, BKM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::max(1, sm_count_gemm() / 2));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    int ncl = 0;
    e = cudaOccupancyMaxActiveClusters(&ncl, (void*)k_ggemm_2sm<kPairStages, BKM>, &cfg);
    if (e != cudaSuccess) return e;
    grid = 2 * std::max(1, ncl);
  }
  if (grid > kMaxGemmCtas) return cudaErrorInvalidConfiguration;  // tensor-map scratch per CTA
  k_ggemm_2sm<kPairStages, BKM><<<grid, kGemmThreads, Cfg::kSmem, st>>>(a, wh, ws, ty, d, sh, p, y);
  return cudaGetLastError();
}

// The CTA-pair weight-gradient kernel on two CTAs per co-resident cluster.
static cudaError_t launch_pair_dw(const Dims& d, const PlanPtrs& p, const CUtensorMap& tx,
                                  const CUtensorMap& tdy, const CUtensorMap& tgh,
                                  const CUtensorMap& tgs, cudaStream_t st) {
  using Cfg = GemmCfgDWPair<kDwPairStages>;
  static int grid = 0;
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(k_ggemm_dw_2sm<kDwPairStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::max(1, sm_count_gemm() / 2));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    int ncl = 0;
    e = cudaOccupancyMaxActiveClusters(&ncl, (void*)k_ggemm_dw_2sm<kDwPairStages>, &cfg);
    if (e != cudaSuccess) return e;
    grid = 2 * std::max(1, ncl);
  }
  if (grid > kMaxGemmCtas) return cudaErrorInvalidConfiguration;  // tensor-map scratch per CTA
  k_ggemm_dw_2sm<kDwPairStages><<<grid, kGemmThreads, Cfg::kSmem, st>>>(tx, tdy, tgh, tgs, d, p);
  return cudaGetLastError();
}

// The two weight tensors as 2D [rows][H'] maps with a box of box_outer rows
// (the input gradient reads them K-major).
static bool encode_weights(const Dims& d, const void* w_home, const void* w_slot,
                           uint32_t box_outer, CUtensorMap* twh, CUtensorMap* tws) {
  if (!encode_2d(twh, w_home, (uint64_t)d.Hp, (uint64_t)d.E * d.H, box_outer)) return false;
  const bool slots = (w_slot != nullptr && d.B > 0);
  return encode_2d(tws, slots ? w_slot : w_home, (uint64_t)d.Hp,
                   slots ? (uint64_t)d.R * d.B * d.H : (uint64_t)d.E * d.H, box_outer);
}

// Forward: Y = recv . W (K = H, N = H', W read N-major).
cudaError_t launch_grouped_gemm(const Dims& d, const PlanPtrs& p, const void* recv,
                                const void* w_home, const void* w_slot, void* y, cudaStream_t st,
                                int* launches) {
  CUtensorMap ta, twh, tws;
  if (!encode_2d(&ta, recv, (uint64_t)d.H, (uint64_t)d.R * d.C, kMmaM)) return cudaErrorInvalidValue;
  const int bn = pick_bn(d.Hp);
  const bool slots = (w_slot != nullptr && d.B > 0);
  if (!encode_panels_3d(&twh, w_home, (uint64_t)d.Hp, (uint64_t)d.E * d.H, bn / 64))
    return cudaErrorInvalidValue;
  if (!encode_panels_3d(&tws, slots ? w_slot : w_home, (uint64_t)d.Hp,
                        slots ? (uint64_t)d.R * d.B * d.H : (uint64_t)d.E * d.H, bn / 64))
    return cudaErrorInvalidValue;
  const long long max_tiles = (long long)d.max_mtiles * (d.Hp / bn);
  const int grid = (int)std::min<long long>(sm_count_gemm(), std::max<long long>(1, max_tiles));
  const GemmShape sh{d.H, d.Hp, d.H};
  cudaError_t e;
  uint16_t* out = (uint16_t*)y;
  if (bn == 256) {
    // 128-row tiles: the single-CTA kernel; 256-row tiles: the CTA-pair kernel
    if (d.tile_m != 2 * kMmaM) {
      e = launch_cfg<GemmCfgM128<256, 4>>(k_ggemm_m128<256, 4, false>, set_fwd128, grid, st, ta, twh,
                                          tws, d, sh, p, out);
      if (e != cudaSuccess) return e;
      *launches += 1;
    }
    if (d.tile_m != kMmaM) {
      CUtensorMap twh2, tws2;  // B halves: 2 panels of 64 columns per CTA
      if (!encode_panels_3d(&twh2, w_home, (uint64_t)d.Hp, (uint64_t)d.E * d.H, 2))
        return cudaErrorInvalidValue;
      if (!encode_panels_3d(&tws2, slots ? w_slot : w_home, (uint64_t)d.Hp,
                            slots ? (uint64_t)d.R * d.B * d.H : (uint64_t)d.E * d.H, 2))
        return cudaErrorInvalidValue;
      e = launch_pair_gemm<false>(d, sh, p, ta, twh2, tws2, out, st);
      if (e != cudaSuccess) return e;
      *launches += 1;
    }
    return cudaSuccess;
  }
  else if (bn == 128) e = launch_bn<128, 6, 4, false>(d, sh, p, ta, twh, tws, out, grid, st, launches);
  else e = launch_bn<64, 8, 5, false>(d, sh, p, ta, twh, tws, out, grid, st, launches);
  return e;
}

// Input gradient: dRecv = dY . W^T (K = H', N = H, W read K-major).
cudaError_t launch_grouped_gemm_dx(const Dims& d, const PlanPtrs& p, const void* dy,
                                   const void* w_home, const void* w_slot, void* d_recv,
                                   cudaStream_t st, int* launches) {
  const int bn = pick_bn(d.H);
  CUtensorMap ta, twh, tws;
  if (!encode_2d(&ta, dy, (uint64_t)d.Hp, (uint64_t)d.R * d.C, kMmaM)) return cudaErrorInvalidValue;
  if (!encode_weights(d, w_home, w_slot, (uint32_t)bn, &twh, &tws)) return cudaErrorInvalidValue;
  const long long max_tiles = (long long)d.max_mtiles * (d.H / bn);
  const int grid = (int)std::min<long long>(sm_count_gemm(), std::max<long long>(1, max_tiles));
  const GemmShape sh{d.Hp, d.H, d.H};
  cudaError_t e;
  uint16_t* out = (uint16_t*)d_recv;
  if (bn == 256) {
    // 128-row tiles: the single-CTA kernel; 256-row tiles: the CTA-pair kernel
    if (d.tile_m != 2 * kMmaM) {
      e = launch_cfg<GemmCfgM128<256, 4>>(k_ggemm_m128<256, 4, true>, set_dx128, grid, st, ta, twh,
                                          tws, d, sh, p, out);
      if (e != cudaSuccess) return e;
      *launches += 1;
    }
    if (d.tile_m != kMmaM) {
      CUtensorMap twh2, tws2;  // B halves: 128 weight rows (n) per CTA
      if (!encode_weights(d, w_home, w_slot, 128, &twh2, &tws2)) return cudaErrorInvalidValue;
      e = launch_pair_gemm<true>(d, sh, p, ta, twh2, tws2, out, st);
      if (e != cudaSuccess) return e;
      *launches += 1;
    }
    return cudaSuccess;
  }
  else if (bn == 128) e = launch_bn<128, 6, 4, true>(d, sh, p, ta, twh, tws, out, grid, st, launches);
  else e = launch_bn<64, 8, 5, true>(d, sh, p, ta, twh, tws, out, grid, st, launches);
  return e;
}

// Weight gradient: G(u,g) += recv[group rows]^T . dY[group rows].
cudaError_t launch_grouped_gemm_dw(const Dims& d, const PlanPtrs& p, const void* recv,
                                   const void* dy, float* g_home, float* g_slot, cudaStream_t st,
                                   int* launches) {
  CUtensorMap tx, tdy, tgh, tgs;
  if (!encode_panels_3d(&tx, recv, (uint64_t)d.H, (uint64_t)d.R * d.C, 2)) return cudaErrorInvalidValue;
  if (!encode_panels_3d(&tdy, dy, (uint64_t)d.Hp, (uint64_t)d.R * d.C, (uint32_t)pick_bn(d.Hp) / 64))
    return cudaErrorInvalidValue;
  // reduce-add targets with a 64-column x 128-row box: 256-byte row segments
  // stream through L2 and DRAM faster than the 128-byte ones of a 32-column box
  const bool slots = g_slot != nullptr && d.B > 0;
  if (!encode_2d_f32_tile(&tgh, g_home, (uint64_t)d.Hp, (uint64_t)d.E * d.H, 64) ||
      !encode_2d_f32_tile(&tgs, slots ? g_slot : g_home, (uint64_t)d.Hp,
                          slots ? (uint64_t)d.R * d.B * d.H : (uint64_t)d.E * d.H, 64))
    return cudaErrorInvalidValue;
  const int bn = pick_bn(d.Hp);
  // L2 prefetch views of G: one box is a whole 128 x BN work-item tile
  CUtensorMap tghp, tgsp;
  if (!encode_2d_f32_tile(&tghp, g_home, (uint64_t)d.Hp, (uint64_t)d.E * d.H, (uint32_t)bn))
    return cudaErrorInvalidValue;
  if (!encode_2d_f32_tile(&tgsp, slots ? g_slot : g_home, (uint64_t)d.Hp,
                          slots ? (uint64_t)d.R * d.B * d.H : (uint64_t)d.E * d.H, (uint32_t)bn))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (bn == 256 && d.H % (2 * kMmaM) == 0) {
    // 256 x 256 work tiles on CTA pairs: each CTA loads 128 of the 256 H' columns of dY
    CUtensorMap tdy2;
    if (!encode_panels_3d(&tdy2, dy, (uint64_t)d.Hp, (uint64_t)d.R * d.C, 2))
      return cudaErrorInvalidValue;
    e = launch_pair_dw(d, p, tx, tdy2, tgh, tgs, st);
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
  const long long max_items = (long long)d.max_groups * (d.H / kMmaM) * (d.Hp / bn);
  const int grid = (int)std::min<long long>(sm_count_gemm(), std::max<long long>(1, max_items));
  if (bn == 256) {
    static bool set = false;
    e = launch_cfg<GemmCfgDW<256, 4>>(k_ggemm_dw<256, 4>, set, grid, st, tx, tdy, tgh, tgs, tghp, tgsp, d, p);
  } else if (bn == 128) {
    static bool set = false;
    e = launch_cfg<GemmCfgDW<128, 5>>(k_ggemm_dw<128, 5>, set, grid, st, tx, tdy, tgh, tgs, tghp, tgsp, d, p);
  } else {
    static bool set = false;
    e = launch_cfg<GemmCfgDW<64, 7>>(k_ggemm_dw<64, 7>, set, grid, st, tx, tdy, tgh, tgs, tghp, tgsp, d, p);
  }
  if (e == cudaSuccess) *launches += 1;
  return e;
}

}  // namespace moonep
