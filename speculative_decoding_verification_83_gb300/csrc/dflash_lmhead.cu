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
// Kernel layout (one CTA per SM, clusters of two CTAs persistent over pairs
// of 128-column vocabulary tiles):
//  * warp 0: TMA producer. Per 32-element step of K it loads its W tile
//    [128 x 32] and half of the h tiles [128 x 32] of the 128-row token
//    tiles, the latter multicast into both CTAs of the cluster, into a
//    five-stage ring (cp.async.bulk.tensor, 64-byte swizzle, mbarrier
//    complete_tx; a stage is reloaded once both CTAs' MMAs have read it);
//  * warp 1: allocates the tensor memory and issues the MMAs from one thread:
//    tcgen05.mma.cta_group::1.kind::f16, M = 128 tokens, N = 128 vocabulary
//    rows, K = 16 per instruction, bf16 in, fp32 accumulated in tensor memory
//    (one 128-column accumulator per token tile, at most four: M <= 512);
//    tcgen05.commit frees a stage when its MMAs have read it, and signals the
//    epilogue after a tile's last step;
//  * warps 2-9: epilogue. Each thread owns one token row of a 32-lane quarter
//    of the accumulators and 64 of a tile's 128 columns (tcgen05.ld.32x32b),
//    rounds the fp32 sums to bf16 (round to nearest even), stores them, and
//    in the fused mode folds them into the row's tile keys (red.max) or
//    argmax (red.max of the (key, index) composite).
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

constexpr int kLmThreads = 320;
constexpr int kBN = 128;                          // vocabulary rows per tile
constexpr int kBK = 32;                           // hidden elements per stage (one 64-byte swizzle row)
constexpr int kMaxMT = kLmMaxRows / 128;          // token tiles
constexpr int kLmStages = 5;
constexpr uint32_t kTileBytes = 128u * kBK * 2u;  // a 128 x 32 bf16 tile, 8 KB
constexpr int kEpiWarp0 = 2;                      // warps 2-9: the epilogue
constexpr int kEpiThreads = kLmThreads - 32 * kEpiWarp0;

struct LmSmem {
  unsigned char a[kLmStages][kMaxMT][kTileBytes];  // h tiles (on 1024-byte boundaries: whole swizzle atoms)
  unsigned char b[kLmStages][kTileBytes];          // W tiles
  uint64_t full[kLmStages], empty[kLmStages];
  uint64_t acc_full, acc_empty;
  uint32_t tmem_base;
  int failed;
  int slot_base[kMaxB];  // per request: its first slot (sampling requests), or -(1 + first slot) (greedy)
  int n_samp;
};
constexpr size_t kLmSmemBytes = sizeof(LmSmem) + 1024;  // + room to align the base to 1024 bytes
static_assert(kLmSmemBytes <= 232448, "one CTA's shared memory (227 KB)");

// ---- PTX wrappers: tensor memory, MMA, TMA --------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, one instruction (M = 128, N = 128, K = 16)
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the mbarrier once the MMAs issued so far have completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
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
// a [128 x 32] bf16 box into the same shared-memory offset of every CTA of
// the cluster in mask, completing bytes on each one's barrier at bar's offset
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* map, int k, int row, uint64_t* bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(k), "r"(row), "r"(smem_addr(bar)), "h"(mask)
      : "memory");
}
// arrive on the barrier at bar's offset in every CTA of mask once this CTA's
// MMAs issued so far have completed
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}
// a [128 x 32] bf16 box of a 2-D tensor map at (k, row) into shared memory
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int k, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(k), "r"(row), "r"(smem_addr(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 64-byte swizzle: rows of 64 bytes (32 bf16 of K), 8-row groups
// 512 bytes apart (stride byte offset), descriptor version 1, swizzle mode 4.
// The leading byte offset is unused in this layout (one MMA's K extent, 32
// bytes, lies inside a swizzle row). Moving along K inside the 64-byte row
// adds the byte offset to the start address.
__device__ __forceinline__ uint64_t sw64_desc(const void* tile) {
  const uint32_t a = smem_addr(tile);
  uint64_t d = (uint64_t)((a & 0x3ffffu) >> 4);
  d |= (uint64_t)1u << 16;           // leading byte offset (unused)
  d |= (uint64_t)(512u >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1u << 46;           // descriptor version
  d |= (uint64_t)4u << 61;           // 64-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ bool lm_wait(uint64_t* bar, uint32_t parity, unsigned long long t0) {
  while (!mbar_try_wait(bar, parity))
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
  const int mt = (p.M + 127) / 128;
  const int n_tiles = (p.V + kBN - 1) / kBN;
  // clusters of two CTAs take pairs of vocabulary tiles (this CTA the one of
  // its rank) and share the h tiles: each loads half of them into both
  const int rank = (int)cluster_rank();
  const int n_pairs = (n_tiles + 1) / 2, pair0 = blockIdx.x / 2, n_clusters = gridDim.x / 2;
  const int nk = p.K / kBK;
  const uint32_t ncols = mt <= 1 ? 128u : (mt <= 2 ? 256u : 512u);

  if (tid == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 2);  // a stage is free once both CTAs' MMAs have read it
    }
    mbar_init(&S.acc_full, 1);
    mbar_init(&S.acc_empty, kEpiThreads);
    S.failed = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&S.tmem_base, ncols);
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
  cluster_sync();  // the peer's barriers are initialised before any load reaches them
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      const unsigned long long t0 = global_timer_ns();
      long long it = 0;
      for (int np = pair0; np < n_pairs && !S.failed; np += n_clusters) {
        const int nt = 2 * np + rank;  // past the last tile for one CTA of an odd pair: W is zero-filled
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = (int)(it % kLmStages);
          const uint32_t ph = (uint32_t)((it / kLmStages) & 1);
          if (it >= kLmStages && !lm_wait(&S.empty[s], ph ^ 1u, t0)) {
            S.failed = 1;
            break;
          }
          mbar_arrive_expect_tx(&S.full[s], (uint32_t)(mt + 1) * kTileBytes);
          tma_load_2d(S.b[s], &map_w, ks * kBK, nt * kBN, &S.full[s]);
          for (int j = rank; j < mt; j += 2) tma_load_2d_mc(S.a[s][j], &map_h, ks * kBK, j * 128, &S.full[s], 3);
        }
      }
      // loads still in flight land before the CTA leaves (bounded)
      const unsigned long long t1 = global_timer_ns();
      for (long long q = it > kLmStages ? it - kLmStages : 0; q < it; ++q)
        (void)lm_wait(&S.full[q % kLmStages], (uint32_t)((q / kLmStages) & 1), t1);
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      const unsigned long long t0 = global_timer_ns();
      long long it = 0;
      int lt = 0;
      for (int np = pair0; np < n_pairs && !S.failed; np += n_clusters, ++lt) {
        if (lt > 0 && !lm_wait(&S.acc_empty, (uint32_t)((lt - 1) & 1), t0)) {
          S.failed = 1;
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < nk; ++ks, ++it) {
          const int s = (int)(it % kLmStages);
          if (!lm_wait(&S.full[s], (uint32_t)((it / kLmStages) & 1), t0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sw64_desc(S.b[s]);
          for (int j = 0; j < mt; ++j) {
            const uint64_t ad = sw64_desc(S.a[s][j]);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)  // 16 elements = 32 bytes = 2 descriptor units
              mma_bf16(tmem + (uint32_t)(j * kBN), ad + 2u * kk, bd + 2u * kk, kIdesc, (ks | kk) != 0 ? 1u : 0u);
          }
          mma_commit_mc(&S.empty[s], 3);  // frees the stage in both CTAs' rings
        }
        if (!ok) {
          S.failed = 1;
          break;
        }
        mma_commit(&S.acc_full);
      }
    }
  } else {
    // ---- epilogue: warps 2-9. Warp w reads lane quarter w % 4 of the
    // accumulators (the lanes a warp may access) and half (w - 2) / 4 of each
    // tile's 128 columns: one 64-logit chunk per row, which is one part of
    // one of the stream's 256-logit tiles
    const int q = warp & 3, hf = (warp - kEpiWarp0) >> 2;
    const unsigned long long t0 = global_timer_ns();
    int lt = 0;
    for (int np = pair0; np < n_pairs; np += n_clusters, ++lt) {
      const int nt = 2 * np + rank;
      const bool ok = lm_wait(&S.acc_full, (uint32_t)(lt & 1), t0);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) S.failed = 1;
        break;
      }
      tc_fence_after();
      const int c0 = nt * kBN + hf * 64;  // this thread's first column
      for (int j = 0; j < mt; ++j) {
        uint32_t ra[32], rb[32];
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(j * kBN + hf * 64);
        tmem_ld32(ta, ra);
        tmem_ld32(ta + 32u, rb);
        tmem_wait_ld();
        const int m = j * 128 + q * 32 + lane;
        const bool row_ok = m < p.M;
        // bf16 pairs, round to nearest even: word i holds columns 2i, 2i + 1
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 x = __float22bfloat162_rn(make_float2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])));
          const __nv_bfloat162 y = __float22bfloat162_rn(make_float2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])));
          pk[i] = *reinterpret_cast<const uint32_t*>(&x);
          pk[16 + i] = *reinterpret_cast<const uint32_t*>(&y);
        }
        const bool whole = c0 + 64 <= p.V;
        if (row_ok && c0 < p.V) {
          uint16_t* out = p.logits + (size_t)m * p.V + c0;
          if (whole) {
            uint4* o4 = reinterpret_cast<uint4*>(out);
#pragma unroll
            for (int v = 0; v < 8; ++v) o4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (c0 + e < p.V) out[e] = (uint16_t)(pk[e >> 1] >> ((e & 1) * 16));
          }
        }
        if (kFused && row_ok && c0 < p.V) {
          // the row's place in the verification: its slot and what the stream
          // would have done with it
          int slot = -1;
          bool greedy = false;
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
          if (slot >= 0 && !greedy) {
            // the chunk's maximum (packed, NaN propagating as in the stream),
            // into tile 4 blk + g: blk its 1024-logit block, g its place in a
            // 256-logit row of that block
            uint32_t key;
            if (whole) {
              __nv_bfloat162 acc = *reinterpret_cast<const __nv_bfloat162*>(&pk[0]);
#pragma unroll
              for (int i = 1; i < 32; ++i) acc = __hmax2_nan(acc, *reinterpret_cast<const __nv_bfloat162*>(&pk[i]));
              key = key_of(max_nan(__low2float(acc), __high2float(acc)));
            } else {
              float mx = -INFINITY;
#pragma unroll
              for (int e = 0; e < 64; ++e)
                if (c0 + e < p.V) mx = max_nan(mx, __uint_as_float((pk[e >> 1] >> ((e & 1) * 16)) << 16));
              key = key_of(mx);
            }
            atomicMax(p.tile_keys + (size_t)slot * p.tiles + (c0 >> 10) * 4 + ((c0 & 255) >> 6), key);
          } else if (greedy) {
            // the lowest column holding the largest key
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
      }
      tc_fence_before();
      mbar_arrive(&S.acc_empty);
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
  cluster_sync();  // no load or arrival of the peer's still reaches this CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
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
// a [rows, K] bf16 row-major matrix read in [128 x 32] boxes, 64-byte swizzle
bool make_map(CUtensorMap* map, const void* base, long long rows, int K) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2u};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, 128u};  // 64 bytes of K: the 64-byte swizzle
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
