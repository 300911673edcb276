// dflash_lmhead.cu -- the target's LM head on the 5th-generation tensor cores,
// with the verification's per-tile statistics in its epilogue.
//
// The draft/verify loop of "DFlash2 用投机解码给 Qwen 提速" (bml.asia) runs the
// target over the prompt plus the block's drafts and reads the logits of
// every position: logits = h W^T, h the positions' last hidden states [M, K]
// and W the vocabulary projection [V, K] (bf16). The verification step then
// reads those logits again. Here the GEMM's epilogue also produces what the
// stream kernel would have computed from them (dflash_sweep.cu): each
// 256-logit tile's maximum as an order key for the top-k rows, and the running
// argmax of the greedy rows. The verification that follows streams nothing
// and runs only its finals (Params::keys_ready), which gather the few
// candidate tiles from the stored logits.
//
// Kernel layout: clusters of two CTAs (one per SM) work as one pair of the
// tensor cores (cta_group::2), persistent over 256-column vocabulary tiles.
// One pair MMA computes D [256 tokens, 256 vocabulary columns] (K = 16):
// each CTA holds the A rows of its 128 tokens and the B rows of its 128
// vocabulary columns, and its tensor memory receives D's rows of its tokens
// over all 256 columns. The tokens come in up to two groups of 256 (M <= 512).
//  * warp 0: TMA producer. Per 64-element step of K each CTA loads its W tile
//    [128 x 64] and its h tile [128 x 64] of each token group into a
//    four-stage ring (cp.async.bulk.tensor, 128-byte swizzle); the bytes of
//    both CTAs complete on the first CTA's barrier, and a stage is reloaded
//    once the pair's MMAs have read it;
//  * warp 1: allocates the pair's tensor memory; in the first CTA, one thread
//    issues the MMAs (tcgen05.mma.cta_group::2.kind::f16, bf16 in, fp32
//    accumulated in tensor memory in two 256-column slots: with one token
//    group the slots alternate between tiles, with two each group has its
//    own, and the next tile's group 0 starts as soon as its slot is read)
//    and the commits that free a stage in both CTAs and signal both
//    epilogues after a tile's last step;
//  * warps 2-13: epilogue. Each thread owns one token row of a 32-lane quarter
//    of its CTA's accumulators and every third 64-column chunk of its groups
//    (tcgen05.ld.32x32b), rounds the fp32 sums to bf16 (round to nearest
//    even), in the fused mode folds them into the row's tile keys (red.max)
//    or argmax (red.max of the (key, index) composite), and stores them,
//    whole 128-byte row segments per store after a transpose in registers.
//    Every epilogue warp of both CTAs reports to the first CTA when it is
//    done with a slot, before its MMAs overwrite the slot.
// Every wait is bounded; a CTA that gives up raises DFLASH_STATUS_TIMEOUT,
// waits (bounded) for its loads in flight and frees its tensor memory.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "dflash_device.cuh"
#include "dflash_internal.h"
#include "dflash_rule.cuh"

namespace dflash {
namespace {

constexpr int kBN = 128;                          // vocabulary rows per CTA (B rows of its half)
constexpr int kPairN = 2 * kBN;                   // vocabulary columns per pair: N of one MMA
constexpr int kGroupM = 256;                      // tokens per group: M of one MMA, 128 per CTA
constexpr int kBK = 64;                           // hidden elements per stage (one 128-byte swizzle row)
constexpr int kMaxG = kLmMaxRows / kGroupM;       // token groups
constexpr int kLmMaxB = kLmMaxRows / 3;           // requests of a fused call (2 gamma + 1 >= 3 rows each)
constexpr int kLmStages = 4;
constexpr uint32_t kTileBytes = 128u * kBK * 2u;  // a 128 x 64 bf16 tile, 16 KB
constexpr int kEpiWarp0 = 2;                      // warps 2-13: the epilogue
constexpr int kEpiWarps = 12;                     // three per lane quarter of the accumulators
constexpr int kEpiSlots = kEpiWarps / 4;
constexpr int kLmThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kEpiThreads = 32 * kEpiWarps;
static_assert(kEpiWarps % 4 == 0, "whole lane quarters");
constexpr int kEpiBarrier = 1;                    // named barrier of the epilogue warps
static_assert(kMaxG * kGroupM == kLmMaxRows, "token groups cover the rows");

struct LmSmem {
  unsigned char b[kLmStages][kTileBytes];          // W tiles (on 1024-byte boundaries: whole swizzle atoms)
  unsigned char a[kLmStages][kMaxG][kTileBytes];   // h tiles of this CTA's tokens
  uint64_t full[kLmStages], empty[kLmStages];
  uint64_t acc_full[2], acc_empty[2];  // per 256-column accumulator slot of the tensor memory
  uint32_t tmem_base;
  int failed;
  int slot_base[kLmMaxB];  // per request: its first slot (sampling requests), or -(1 + first slot) (greedy)
  int n_samp;
};
constexpr size_t kLmSmemBytes = sizeof(LmSmem) + 1024;  // + room to align the base to 1024 bytes
static_assert(kLmSmemBytes <= 232448, "one CTA's shared memory (227 KB)");

// ---- PTX wrappers: tensor memory, MMA, TMA, cluster barriers ---------------------------
// Every tcgen05 instruction of the kernel that names a CTA group names the
// pair (cta_group::2): allocation and release are made by one warp of each
// CTA together, the MMAs and their commits by one thread of the first CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem of both CTAs] (+)= A[smem desc, both CTAs] * B[smem desc, both CTAs]^T:
// one pair instruction, M = 256 (128 rows per CTA), N = 256 (128 B rows per CTA), K = 16
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at bar's offset in every CTA of mask once the pair
// MMAs issued so far have completed
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}
// 32 consecutive fp32 columns of this thread's lane (completes at tmem_wait_ld)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// this CTA's rank in its cluster, and a barrier over the cluster's threads
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the cluster-window address of the same shared-memory object in the first CTA
__device__ __forceinline__ uint32_t first_cta_addr(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_addr(p)));
  return r;
}
// a [128 x 64] bf16 box of a 2-D tensor map at (k, row) into this CTA's shared
// memory, its bytes completing on a barrier of either CTA of the pair
__device__ __forceinline__ void tma_load_pair(void* dst, const CUtensorMap* map, int k, int row,
                                              uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(k), "r"(row), "r"(bar_cluster)
      : "memory");
}
// arrive on a barrier of another CTA of the cluster
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// a wait that also orders what the other CTA of the pair did before it arrived
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}
// the epilogue warps' own barrier: the AND of every epilogue thread's flag
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kEpiBarrier), "n"(kEpiThreads)
      : "memory");
  return r != 0u;
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 bytes (64 bf16 of K), 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1, swizzle mode 2.
// The leading byte offset is unused in this layout (one MMA's K extent, 32
// bytes, lies inside a swizzle row). Moving along K inside the 128-byte row
// adds the byte offset to the start address. In a pair MMA the same offset
// addresses each CTA's own tile.
__device__ __forceinline__ uint64_t sw128_desc(const void* tile) {
  const uint32_t a = smem_addr(tile);
  uint64_t d = (uint64_t)((a & 0x3ffffu) >> 4);
  d |= (uint64_t)1u << 16;            // leading byte offset (unused)
  d |= (uint64_t)(1024u >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1u << 46;            // descriptor version
  d |= (uint64_t)2u << 61;            // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 256, M = 256 (the pair's rows).
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kPairN >> 3) << 17) | ((uint32_t)(kGroupM >> 4) << 24);

// Inside each group of 8 lanes, lane t holds the eight 16-byte pieces of row
// t (piece p in words 4p..4p+3); afterwards it holds piece t of the group's
// row i in words 4i..4i+3. Three butterfly stages (lane masks 4, 2, 1) each
// swap the four pieces whose index differs from the lane's in that bit.
__device__ __forceinline__ void transpose_pieces8(uint32_t (&pk)[32], int lane) {
#pragma unroll
  for (int b = 2; b >= 0; --b) {
    const int m = 1 << b;
    const bool hi = (lane & m) != 0;
#pragma unroll
    for (int s0 = 0; s0 < 8; ++s0) {
      if (s0 & m) continue;
      const int s1 = s0 | m;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi ? pk[4 * s0 + w] : pk[4 * s1 + w], m);
        if (hi)
          pk[4 * s0 + w] = recv;
        else
          pk[4 * s1 + w] = recv;
      }
    }
  }
}

// Bounded waits: each gives up kWaitLimitNs after it began (a long GEMM
// makes progress between its waits); lm_wait_from counts from t0, so that
// several waits share one limit.
__device__ __forceinline__ bool lm_wait_from(uint64_t* bar, uint32_t parity, unsigned long long t0) {
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
__device__ __forceinline__ bool lm_wait(uint64_t* bar, uint32_t parity) {
  return mbar_try_wait(bar, parity) || lm_wait_from(bar, parity, global_timer_ns());
}
__device__ __forceinline__ bool lm_wait_cluster(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait_cluster(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// ---- the kernel ----------------------------------------------------------------------------
template <bool kFused>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                  const LmParams p) {
  extern __shared__ unsigned char lm_raw[];
  LmSmem& S = *reinterpret_cast<LmSmem*>((reinterpret_cast<uintptr_t>(lm_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int groups = (p.M + kGroupM - 1) / kGroupM;
  // each cluster is one pair of the tensor cores over 256-column vocabulary
  // tiles: this CTA holds the W rows of its half of the tile and the h rows
  // of its half of each token group
  const int rank = (int)cluster_rank();
  const int n_pairs = (p.V + kPairN - 1) / kPairN, pair0 = blockIdx.x / 2, n_clusters = gridDim.x / 2;
  const int nk = p.K / kBK;
  // Tensor memory: two 256-column accumulator slots. With one token group
  // they alternate between vocabulary tiles, so the epilogue of one tile runs
  // while the MMAs of the next fill the other slot; with two groups each
  // group has its slot, released as soon as the epilogue has read it.
  const uint32_t ncols = 512u;

  if (tid == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      mbar_init(&S.full[s], 1);   // the first CTA's producer; both CTAs' bytes
      mbar_init(&S.empty[s], 1);  // the pair's commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&S.acc_full[a], 1);
      mbar_init(&S.acc_empty[a], 2 * kEpiWarps);  // every epilogue warp of both CTAs
    }
    S.failed = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(&S.tmem_base, ncols);
  if (kFused) {
    // slots of the verification (sampling requests first, in request order,
    // 2 gamma + 1 slots each; then greedy requests, gamma + 1 each): each
    // thread counts the sampling requests of its run of requests, a block
    // scan gives every run its ordinals
    const int chunk = (p.B + kLmThreads - 1) / kLmThreads;
    const int lo = min(p.B, tid * chunk), hi = min(p.B, lo + chunk);
    int mine = 0;
    for (int b = lo; b < hi; ++b) mine += sampling_temperature(__ldg(p.temperature + b)) ? 1 : 0;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    __shared__ int warp_tot[kLmThreads / 32];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = incl - mine, ns = 0;
    for (int w = 0; w < kLmThreads / 32; ++w) {
      if (w < warp) before += warp_tot[w];
      ns += warp_tot[w];
    }
    int os = before, og = lo - before;
    for (int b = lo; b < hi; ++b) {
      if (sampling_temperature(__ldg(p.temperature + b)))
        S.slot_base[b] = (os++) * (2 * p.gamma + 1);
      else
        S.slot_base[b] = -1 - (ns * (2 * p.gamma + 1) + (og++) * (p.gamma + 1));
    }
    if (tid == 0) S.n_samp = ns;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any load or arrival reaches them
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // the verification launched after this kernel may be scheduled as SMs free
  // up; it waits for this grid's completion before reading what it wrote
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ---- TMA producer (both CTAs)
    if (lane == 0) {
      long long it = 0;
      for (int np = pair0; np < n_pairs && !S.failed; np += n_clusters) {
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = (int)(it % kLmStages);
          const uint32_t ph = (uint32_t)((it / kLmStages) & 1);
          if (it >= kLmStages && !lm_wait(&S.empty[s], ph ^ 1u)) {
            S.failed = 1;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&S.full[s], 2u * (uint32_t)(groups + 1) * kTileBytes);
          const uint32_t bar = first_cta_addr(&S.full[s]);
          // rows past the end of W or h (a last half tile, a last token group) are zero-filled
          tma_load_pair(S.b[s], &map_w, ks * kBK, np * kPairN + rank * kBN, bar);
          for (int j = 0; j < groups; ++j)
            tma_load_pair(S.a[s][j], &map_h, ks * kBK, j * kGroupM + rank * 128, bar);
        }
      }
      // every load issued has landed once the MMAs that read it have
      // completed and freed its stage (bounded)
      const unsigned long long t1 = global_timer_ns();
      for (long long q = it > kLmStages ? it - kLmStages : 0; q < it; ++q)
        (void)lm_wait_from(&S.empty[q % kLmStages], (uint32_t)((q / kLmStages) & 1), t1);
    }
  } else if (warp == 1) {
    // ---- MMA issuer (the first CTA, for the pair)
    if (lane == 0 && rank == 0) {
      long long it = 0;
      int lt = 0;
      // this step's MMAs of group j into accumulator slot `slot`
      auto mma_step = [&](int s, int j, int slot, int ks) {
        const uint64_t bd = sw128_desc(S.b[s]), ad = sw128_desc(S.a[s][j]);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)  // 16 elements = 32 bytes = 2 descriptor units
          mma_pair(tmem + (uint32_t)(slot * kPairN), ad + 2u * kk, bd + 2u * kk, kIdesc, (ks | kk) != 0 ? 1u : 0u);
      };
      auto stage_full = [&](long long i) {
        const bool ok = lm_wait(&S.full[i % kLmStages], (uint32_t)((i / kLmStages) & 1));
        tc_fence_after();
        return ok;
      };
      bool ok = true;
      for (int np = pair0; np < n_pairs && ok; np += n_clusters, ++lt) {
        if (groups == 1) {
          // one group: the slots alternate; slot lt % 2 was last read by the
          // epilogue of tile lt - 2
          const int slot = lt & 1, use = lt >> 1;
          if (use > 0 && !lm_wait_cluster(&S.acc_empty[slot], (uint32_t)((use - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int ks = 0; ks < nk && ok; ++ks, ++it) {
            if (!(ok = stage_full(it))) break;
            mma_step((int)(it % kLmStages), 0, slot, ks);
            mma_commit_pair(&S.empty[it % kLmStages], 3);  // frees the stage in both CTAs' rings
          }
          if (ok) mma_commit_pair(&S.acc_full[slot], 3);  // both CTAs' accumulators are complete
        } else {
          // two groups, slot j for group j: the first ring's worth of steps
          // goes to group 0 as soon as its slot is read, then group 1 catches
          // up on the same stages once its slot is read too
          if (lt > 0 && !lm_wait_cluster(&S.acc_empty[0], (uint32_t)((lt - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int head = nk < kLmStages ? nk : kLmStages;
          for (int ks = 0; ks < head && ok; ++ks)
            if ((ok = stage_full(it + ks))) mma_step((int)((it + ks) % kLmStages), 0, 0, ks);
          if (ok && lt > 0 && !lm_wait_cluster(&S.acc_empty[1], (uint32_t)((lt - 1) & 1))) ok = false;
          if (!ok) break;
          tc_fence_after();
          for (int ks = 0; ks < head; ++ks) {
            mma_step((int)((it + ks) % kLmStages), 1, 1, ks);
            mma_commit_pair(&S.empty[(it + ks) % kLmStages], 3);
          }
          it += head;
          for (int ks = head; ks < nk && ok; ++ks, ++it) {
            if (!(ok = stage_full(it))) break;
            const int s = (int)(it % kLmStages);
            mma_step(s, 0, 0, ks);
            mma_step(s, 1, 1, ks);
            mma_commit_pair(&S.empty[s], 3);
          }
          if (ok) mma_commit_pair(&S.acc_full[0], 3);  // both groups, both CTAs
        }
      }
      if (!ok) S.failed = 1;
    }
  } else {
    // ---- epilogue: warps 2-13. Warp w reads lane quarter w % 4 of this CTA's
    // accumulators (the lanes a warp may access) and every third of the
    // quarter's 64-column chunks from (w - 2) / 4 on: each chunk one part of
    // one of the stream's 256-logit tiles
    const int q = warp & 3, es = (warp - kEpiWarp0) >> 2;
    int lt = 0;
    // one arrival per warp and slot use on the first CTA's barrier, before
    // its MMAs overwrite the slot
    auto release = [&](int slot) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&S.acc_empty[slot]);
        else
          mbar_arrive_cluster(first_cta_addr(&S.acc_empty[slot]));
      }
    };
    for (int np = pair0; np < n_pairs; np += n_clusters, ++lt) {
      const int slot1 = lt & 1;  // one group: this tile's slot
      const bool ok = groups == 1 ? lm_wait(&S.acc_full[slot1], (uint32_t)((lt >> 1) & 1))
                                  : lm_wait(&S.acc_full[0], (uint32_t)(lt & 1));
      if (!epi_all(ok)) {
        if (tid == kEpiWarp0 * 32) S.failed = 1;
        break;
      }
      tc_fence_after();
      // the quarter's 64-column chunks (four per token group), dealt to its
      // kEpiSlots warps in turn
      for (int ci = es; ci < 4 * groups; ci += kEpiSlots) {
        const int j = ci >> 2, cc = ci & 3;
        const int acc = groups == 1 ? slot1 : j;  // the accumulator slot
        const int m0 = j * kGroupM + rank * 128 + q * 32;
        // with two groups, group 0's slot is released after the warp's last
        // chunk of it (every warp has one: es < 4)
        const bool last_of_group0 = groups == 2 && ci < 4 && ci + kEpiSlots >= 4;
        if (m0 >= p.M) {  // the warp's rows are past the last token
          if (last_of_group0) release(0);
          continue;
        }
        const int m = m0 + lane;
        const bool row_ok = m < p.M;
        // the row's place in the verification: its slot and what the stream
        // would have done with it
        int slot = -1;
        bool greedy = false;
        if (kFused && row_ok) {
          const int g1 = p.gamma + 1;
          if (m < p.Mt) {
            const int b = m / g1, i = m - b * g1;
            const int base = S.slot_base[b];
            if (base >= 0) {
              slot = base + 2 * i;
            } else {
              slot = -1 - base + i;
              greedy = true;
            }
          } else {
            const int b = (m - p.Mt) / p.gamma, i = (m - p.Mt) - b * p.gamma;
            const int base = S.slot_base[b];
            if (base >= 0) slot = base + 2 * i + 1;  // a greedy request reads no draft rows
          }
        }
        {
          uint32_t ra[32], rb[32];
          const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kPairN + cc * 64);
          tmem_ld32(ta, ra);
          tmem_ld32(ta + 32u, rb);
          tmem_wait_ld();
          const int c0 = np * kPairN + cc * 64;  // this thread's first column
          // bf16 pairs, round to nearest even: word i holds columns 2i, 2i + 1
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 x =
                __float22bfloat162_rn(make_float2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])));
            const __nv_bfloat162 y =
                __float22bfloat162_rn(make_float2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])));
            pk[i] = *reinterpret_cast<const uint32_t*>(&x);
            pk[16 + i] = *reinterpret_cast<const uint32_t*>(&y);
          }
          const bool whole = c0 + 64 <= p.V;
          if (kFused && row_ok && c0 < p.V && slot >= 0) {
            // the chunk's maximum (packed, NaN propagating as in the stream)
            float mx = -INFINITY;
            if (whole) {
              __nv_bfloat162 acc = *reinterpret_cast<const __nv_bfloat162*>(&pk[0]);
#pragma unroll
              for (int i = 1; i < 32; ++i) acc = __hmax2_nan(acc, *reinterpret_cast<const __nv_bfloat162*>(&pk[i]));
              mx = max_nan(__low2float(acc), __high2float(acc));
            } else {
#pragma unroll
              for (int e = 0; e < 64; ++e)
                if (c0 + e < p.V) mx = max_nan(mx, __uint_as_float((pk[e >> 1] >> ((e & 1) * 16)) << 16));
            }
            if (!greedy) {
              // into tile 4 blk + g: blk its 1024-logit block, g its place in
              // a 256-logit row of that block
              atomicMax(p.tile_keys + (size_t)slot * p.tiles + (c0 >> 10) * 4 + ((c0 & 255) >> 6), key_of(mx));
            } else if (whole && !isnan(mx)) {
              // the lowest column holding the maximum (-0 equal to +0, as in
              // the key order; no NaN in the chunk)
              const __nv_bfloat162 m2 = __float2bfloat162_rn(mx);  // exact: mx is a bf16 value
              int col = 0;
#pragma unroll
              for (int i = 31; i >= 0; --i) {
                const uint32_t eq = __heq2_mask(*reinterpret_cast<const __nv_bfloat162*>(&pk[i]), m2);
                col = (eq & 0xffffu) ? 2 * i : (eq ? 2 * i + 1 : col);
              }
              red_max_gpu(p.row_best + slot, composite(key_of(mx), c0 + col));
            } else {
              // a NaN in the chunk, or its last columns past the end: the key
              // order decides, element by element
              uint32_t best = 0u;
              int col = 0;
#pragma unroll
              for (int e = 0; e < 64; ++e) {
                const uint32_t k = c0 + e < p.V ? key_of(__uint_as_float((pk[e >> 1] >> ((e & 1) * 16)) << 16)) : 0u;
                if (k > best) {
                  best = k;
                  col = c0 + e;
                }
              }
              if (best) red_max_gpu(p.row_best + slot, composite(best, col));
            }
          }
          if (whole) {
            // whole 128-byte rows per store: after the transpose the lanes of
            // each 8-lane group write the eight pieces of one of its rows
            transpose_pieces8(pk, lane);
            const int r0 = m0 + (lane & ~7), t8 = lane & 7;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (r0 + i < p.M)
                *reinterpret_cast<uint4*>(p.logits + (size_t)(r0 + i) * p.V + c0 + 8 * t8) =
                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          } else if (row_ok && c0 < p.V) {
            uint16_t* out = p.logits + (size_t)m * p.V + c0;
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (c0 + e < p.V) out[e] = (uint16_t)(pk[e >> 1] >> ((e & 1) * 16));
          }
        }
        if (last_of_group0) release(0);
      }
      release(groups == 1 ? slot1 : 1);  // the warp is done with this tile's (last) slot
    }
  }

  if (kFused && blockIdx.x == 0 && warp >= kEpiWarp0) {
    // Tiles with no logit (past the row's end, inside its last 16 KB piece):
    // the stream writes the key of -inf for them, and the finals wait for
    // every key of a row to be non-zero.
    const int first = ((p.V + 1023) >> 10) * 4;  // whole 1024-logit blocks past the end
    const int partial_blk = p.V >> 10, rem = p.V & 1023;
    const int n_topk_slots = S.n_samp * (2 * p.gamma + 1);
    for (int slot = tid - kEpiWarp0 * 32; slot < n_topk_slots; slot += kEpiThreads) {
      uint32_t* keys = p.tile_keys + (size_t)slot * p.tiles;
      for (int t = first; t < p.tiles; ++t) keys[t] = kKeyNegInf;
      if (rem)  // tiles of the last block whose four 64-logit chunks all lie past the end
        for (int g = 0; g < 4; ++g)
          if (g * 64 >= rem) keys[partial_blk * 4 + g] = kKeyNegInf;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no load, commit or arrival of the pair still reaches either CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, ncols);
  }
  if (tid == 0 && S.failed && p.status) atomicOr(p.status, kStatusTimeout);
}

// ---- host: tensor maps ------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}
// a [rows, K] bf16 row-major matrix read in [128 x 64] boxes, 128-byte swizzle
bool make_map(CUtensorMap* map, const void* base, long long rows, int K) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2u};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, 128u};  // 128 bytes of K: the 128-byte swizzle
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int lmhead_smem_bytes() { return (int)kLmSmemBytes; }

int launch_lmhead(const LmParams& p, const void* h, const void* w, bool fused, int grid, void* stream) {
  CUtensorMap mw, mh;
  if (!make_map(&mw, w, p.V, p.K) || !make_map(&mh, h, p.M, p.K)) return (int)cudaErrorInvalidValue;
  static bool ready[kMaxDevices][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  if (!ready[dev][fused ? 1 : 0]) {
    e = fused ? cudaFuncSetAttribute(lmhead_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kLmSmemBytes)
              : cudaFuncSetAttribute(lmhead_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kLmSmemBytes);
    if (e != cudaSuccess) return (int)e;
    ready[dev][fused ? 1 : 0] = true;
  }
  // clusters of two CTAs (an even grid: two SMs a cluster)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid < 2 ? 2 : grid & ~1));
  cfg.blockDim = dim3(kLmThreads);
  cfg.dynamicSmemBytes = kLmSmemBytes;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)(fused ? cudaLaunchKernelEx(&cfg, lmhead_kernel<true>, mw, mh, p)
                     : cudaLaunchKernelEx(&cfg, lmhead_kernel<false>, mw, mh, p));
}

}  // namespace dflash
