// Iteration smoothing (kernel "b"; dInfer explainer, diffusion-iteration manager): the rows left
// undecided after this step's commit feed the next round with their whole distribution,
//   S[j, :] = sum_v bf16(exp(z_{r_j, v} - lse_{r_j})) * E[v, :].
//
// prob_rows_kernel writes the bf16 probability rows P (compacted; the single-read step writes
// them from its statistics kernel instead), then smooth_gemm_kernel contracts P with the
// embedding table on the 5th-generation tensor cores (and splitk_reduce_kernel adds the split-K
// partial sums, in a fixed order, when the plan splits K).
// Both operands are stored K-slab-blocked, [ceil(V/64)][rows][64]: the 64-wide K slab of every
// row is contiguous, so the 128 rows a CTA needs from one slab are one contiguous 16 KB run.
// TMA (3-D tensor maps over the blocked layout, 128-byte swizzle; two slabs per box) brings
// those runs into a multi-stage shared-memory ring; tcgen05.mma accumulates in TMEM; epilogue
// warps read the accumulator back with tcgen05.ld.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "mbarrier.cuh"
#include "vec_math.cuh"

namespace dllm {
namespace {

// ------------------------------------------------------------------ PTX wrappers

// TMA box (0, y, slab) of a K-slab-blocked operand (rows y.. of one 64-wide K slab) into this
// CTA's shared memory.  .cta_group::2: the completion may be signalled on an mbarrier in either
// CTA of the pair (`bar` is a shared::cluster address); both CTAs' boxes complete on the leader's
// barrier, so no thread has to relay the peer's progress.
__device__ __forceinline__ void tma_load_slab_pair(uint32_t dst, const CUtensorMap* map,
                                                   uint32_t bar, int y, int slab) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(y), "r"(slab)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
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

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Pair MMA issued by the leader CTA: D[256 x N] (+)= A[256 x 16] * B[N x 16]^T, bf16 inputs,
// fp32 accumulators.  Each CTA holds 128 rows of A and N/2 rows of B at the same shared-memory
// offsets, and receives its own 128 rows of D in its tensor memory.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at offset `bar` in both CTAs of the pair once every tcgen05 operation
// issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows 128 B apart,
// 8-row groups 1024 B apart: 16-byte chunk c of row i at i * 128 + ((c ^ (i & 7)) * 16).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor: dense, D fp32, A and B bf16, both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing ever arrives at;
// after limit_ns the wait gives up and records DLLM_ERR_TIMEOUT in the status word.
__global__ void wait_timeout_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bar(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

// ------------------------------------------------------------------ GEMM

constexpr int kBM = 128;   // rows per CTA; a CTA pair covers 256
constexpr int kBK = 64;    // one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;
constexpr int kGemmThreads = 256;  // warp 0: TMEM allocation + MMA issue (leader);
                                   // warps 1-7: producers, one ring stage each;
                                   // warps 4-7 then drain the accumulator (epilogue)
constexpr int kProducers = 7;
constexpr int kATileBytes = kBM * kBK * 2;
constexpr int kMaxStages = 8;

struct GemmParams {
  CUtensorMap tmA;    // P: K-slab-blocked [slabs][R_pad][64], boxes of 64 x 128 x gs
  CUtensorMap tmB;    // E^T: K-slab-blocked [slabs][d][64], boxes of 64 x bn_max/2 x gs
  int num_kb;         // 64-wide K blocks over V
  int n_tiles;
  int bn_base;        // narrow pair-tile width; the first bn_rem tiles are 16 wider
  int bn_rem;
  int bn_max;
  int split_k;        // K splits of the main pairs (their partial sums 0 .. split_k - 1)
  int kb_per_split;   // K blocks of each main split
  int main_pairs;     // pairs [0, main_pairs): one tile over one K split each
  int tail_pairs;     // pairs after them: tail_tiles tiles each over the tail K range
  int tail_tiles;
  int kb_tail0;       // first K block of the tail range (the tail's partial sum is split_k)
  int stages;
  int gs;             // K slabs per stage
  int tmem_cols;
  int acc_cols;       // TMEM columns between the two accumulators (0: one accumulator)
  int d;
  int R_pad;
  float* out;          // [M, d] when there is a single K range
  float* part;         // [partials, R_pad, d] otherwise
  const int32_t* M;
  const int32_t* row_map;  // out row of P row j (-1: skipped); null: j itself
  int32_t* status;
  int wait_late;           // P and M come from earlier kernels than the one just before this
                           // one, which only writes the row map: wait for it in the epilogue
};

// Bounded wait with acquire at cluster scope (the barrier is arrived at from both CTAs of the
// pair, after their tensor-memory reads).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity,
                                                 volatile int* abort_flag, int32_t* status) {
  uint64_t t0 = 0;
  for (uint32_t spins = 0;; ++spins) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((spins & 1023u) == 1023u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        set_status(status, DLLM_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// One tile of a CTA pair's work: rows m0.. (256), columns n0.. (bn), K blocks kb0.. (nkb),
// written to partial sum `part_idx` (or straight to the output).
struct GemmUnit {
  int m0, n0, bn, kb0, nkb, part_idx;
};

__device__ __forceinline__ GemmUnit gemm_unit(const GemmParams& p, int pair, int u) {
  GemmUnit w;
  int tile;
  if (pair < p.main_pairs) {
    const int ks = pair % p.split_k;
    tile = pair / p.split_k;
    w.kb0 = ks * p.kb_per_split;
    const int end = p.tail_pairs > 0 ? p.kb_tail0 : p.num_kb;
    w.nkb = max(0, min(end, w.kb0 + p.kb_per_split) - w.kb0);
    w.part_idx = ks;
  } else {
    tile = (pair - p.main_pairs) * p.tail_tiles + u;
    w.kb0 = p.kb_tail0;
    w.nkb = p.num_kb - p.kb_tail0;
    w.part_idx = p.split_k;
  }
  const int n_tile = tile % p.n_tiles;
  w.m0 = (tile / p.n_tiles) * 2 * kBM;
  w.n0 = n_tile * p.bn_base + min(n_tile, p.bn_rem) * 16;
  w.bn = p.bn_base + (n_tile < p.bn_rem ? 16 : 0);
  return w;
}

// A CTA pair (a 2-CTA cluster) computes 256 x BN tiles of S over K ranges: a main pair one
// tile over one of split_k equal K ranges; a tail pair (the pairs that would otherwise leave
// SMs idle) a run of tail_tiles tiles, each over the last, short K range, so that every pair
// of the grid streams about the same number of K blocks.  Both CTAs stream their own 128 rows
// of P and their own BN/2 rows of E^T through a `stages`-deep ring whose stages hold `gs`
// consecutive 64-wide K slabs of each operand (one TMA box each), one continuous sequence of
// stages over the pair's tiles.  Producer warps issue a stage's two TMA boxes in their CTA
// once the stage is free, and both CTAs' boxes complete on the leader CTA's "full" barrier for
// that stage (the leader's producer posts the byte count of all four boxes).  The leader's MMA
// thread issues tcgen05.mma.cta_group::2 (M = 256, N = BN) into one of two TMEM accumulators
// (alternating by tile), multicasts each stage's release and each tile's accumulator-ready
// signal to both CTAs; the four epilogue warps of each CTA drain a finished accumulator while
// the MMAs of the next tile run into the other, and release it on the leader's barrier.  No
// thread relays ring progress across the pair: an earlier version in which the peer's stages
// were forwarded by a cluster-scope release arrive spent ~0.7 us per stage on that hop.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    smooth_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t dyn_raw[];
  __shared__ uint64_t bars[2 * kMaxStages + 5];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int m_pairs = p.R_pad / (2 * kBM);
  const int n_units = pair < p.main_pairs
                          ? 1
                          : min(p.tail_tiles, m_pairs * p.n_tiles -
                                                  (pair - p.main_pairs) * p.tail_tiles);
  // P, M and the row map come from the kernels before this one.  With wait_late (the
  // single-read step), the kernel just before writes the row map and lets this grid launch
  // before it waits for the commit kernel ahead of it; that commit kernel waited for the
  // statistics grid before it let the map kernel launch, so P and M (written further back) are
  // complete when this grid starts, and only the row map is waited for, by the epilogue, while
  // the mainloop overlaps the commit and map kernels.
  if (!p.wait_late) pdl_wait();
  pdl_trigger();
  const int Mdev = *reinterpret_cast<const volatile int32_t*>(p.M);
  // tiles whose rows are all beyond M are skipped (they come last in a pair's run)
  int U = 0;
  while (U < n_units && gemm_unit(p, pair, U).m0 < Mdev) ++U;
  if (U == 0) {
    // both CTAs of the pair leave together: no row of the pair is kept.  With wait_late this
    // CTA still waits for the kernel before it: the next launch on the stream waits only for
    // this grid, so no CTA may finish before the row map (and the block state it reads) is
    // final, or a following reset could rewrite that state while the map still reads it.
    if (p.wait_late) pdl_wait();
    return;
  }
  const int S = p.stages;
  const int P = min(S, p.acc_cols > 0 ? 3 : kProducers);  // producers: warps 1..P
  const int G = p.gs;
  const int nst1 = (gemm_unit(p, pair, 0).nkb + G - 1) / G;  // ring stages per tile
  const int nst = U * nst1;
  const bool direct = p.split_k == 1 && p.tail_pairs == 0;  // no partial sums
  const uint32_t b_half_bytes = static_cast<uint32_t>(p.bn_max / 2) * kBK * 2;
  const uint32_t a_stage = static_cast<uint32_t>(G) * kATileBytes;
  const uint32_t b_stage = static_cast<uint32_t>(G) * b_half_bytes;

  const uint32_t raw = smem_u32(dyn_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + S * a_stage;
  const uint32_t full0 = smem_u32(&bars[0]);
  const uint32_t empty0 = smem_u32(&bars[kMaxStages]);
  const uint32_t accf0 = smem_u32(&bars[2 * kMaxStages]);      // accumulator a ready: + 8a
  const uint32_t acce0 = smem_u32(&bars[2 * kMaxStages + 2]);  // accumulator a drained: + 8a
  const uint32_t done_bar = smem_u32(&bars[2 * kMaxStages + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);  // the leader producer's expect-tx arrival (the peer's
                                    // full barriers are not used)
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, 8);  // the four epilogue warps of both CTAs (leader's is used)
    }
    mbar_init(done_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(smem_u32(&tmem_slot), p.tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anyone signals across the pair
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_v = &abort_flag;
  const int prod = warp - 1;  // producer index of warps 1..P

  int last_k = -1;  // this producer's last issued stage (drained after an abort)
  if (warp >= 1 && prod < P) {
    // ---- producers (both CTAs): stages prod, prod + P, ... of own 128 P rows and own half
    // of the E^T tile; whole warps wait, lane 0 issues.  A box reaching past the last slab
    // reads zeros there and still counts its full size.
    const uint32_t leader_full0 = map_to_rank(full0, 0);
    const uint32_t stage_tx = 2u * (a_stage + b_stage);
    if (lane == 0) {
      prefetch_tensormap(&p.tmA);
      prefetch_tensormap(&p.tmB);
    }
    // this producer's position: stage kk of tile u; the tile's coordinates are worked out
    // once per tile, never between a stage's release and its refill
    int u = 0, kk = prod;
    GemmUnit w = gemm_unit(p, pair, 0);
    int ya = w.m0 + static_cast<int>(rank) * kBM, yb = w.n0 + static_cast<int>(rank) * (w.bn / 2);
    for (int k = prod; k < nst; k += P, kk += P) {
      while (kk >= nst1) {
        kk -= nst1;
        w = gemm_unit(p, pair, ++u);
        ya = w.m0 + static_cast<int>(rank) * kBM;
        yb = w.n0 + static_cast<int>(rank) * (w.bn / 2);
      }
      const int slab = w.kb0 + kk * G;
      const int s = k % S;
      const uint32_t ph = (k / S) & 1;
      if (!__all_sync(kFull, wait_bar(empty0 + 8 * s, ph ^ 1, abort_v, p.status))) break;
      if (lane == 0) {
        if (leader) mbar_expect_tx(full0 + 8 * s, stage_tx);
        tma_load_slab_pair(sA + s * a_stage, &p.tmA, leader_full0 + 8 * s, ya, slab);
        tma_load_slab_pair(sB + s * b_stage, &p.tmB, leader_full0 + 8 * s, yb, slab);
      }
      last_k = k;
      __syncwarp();
    }
  } else if (warp == 0 && lane == 0 && leader) {
    // ---- MMA issuer (leader): tile u into accumulator u % 2
    bool ok = true;
    for (int u = 0; u < U && ok; ++u) {
      const int a = u & 1;
      // the epilogue warps of both CTAs have drained this accumulator's previous tile
      if (u >= 2 && !wait_bar_cluster(acce0 + 8 * a, ((u >> 1) - 1) & 1, abort_v, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const GemmUnit w = gemm_unit(p, pair, u);
      const uint32_t idesc = idesc_bf16(2 * kBM, w.bn);
      const uint32_t d_tmem = tmem + static_cast<uint32_t>(a * p.acc_cols);
      for (int kk = 0; kk < nst1; ++kk) {
        const int k = u * nst1 + kk;
        const int s = k % S;
        const uint32_t ph = (k / S) & 1;
        if (!wait_bar(full0 + 8 * s, ph, abort_v, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nv = min(G, w.nkb - kk * G);  // slabs of this stage inside the tile's K range
        for (int g = 0; g < nv; ++g) {
          const uint32_t a_s = sA + s * a_stage + g * kATileBytes;
          const uint32_t b_s = sB + s * b_stage + g * b_half_bytes;
#pragma unroll
          for (int k2 = 0; k2 < kBK / kUmmaK; ++k2) {
            umma_bf16_pair(d_tmem, sw128_desc(a_s + k2 * kUmmaK * 2),
                           sw128_desc(b_s + k2 * kUmmaK * 2), idesc,
                           (kk > 0 || g > 0 || k2 > 0) ? 1u : 0u);
          }
        }
        umma_commit_pair(empty0 + 8 * s);  // stage s is free in both CTAs once these MMAs read it
      }
      if (ok) umma_commit_pair(accf0 + 8 * a);  // tile u's accumulator complete in both CTAs
    }
    umma_commit_pair(done_bar);  // every MMA issued so far has completed
  }
  if (warp >= 4) {
    // ---- epilogue (both CTAs): this CTA's 128 rows of each finished tile, TMEM -> registers ->
    // global, then the accumulator is released to the leader's MMA thread
    if (p.wait_late) pdl_wait();  // the row map and the output buffers
    __syncwarp();
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    for (int u = 0; u < U; ++u) {
      const int a = u & 1;
      // warp-uniform: tcgen05.ld below is a .sync.aligned warp instruction
      const bool ok = __all_sync(kFull, wait_bar(accf0 + 8 * a, (u >> 1) & 1, abort_v, p.status));
      tc_fence_after();
      if (!ok) break;
      const GemmUnit w = gemm_unit(p, pair, u);
      const int row = w.m0 + static_cast<int>(rank) * kBM + q * 32 + lane;
      float* dst_base =
          direct ? p.out : p.part + static_cast<size_t>(w.part_idx) * p.R_pad * p.d;
      // partial sums keep P's row order; the final rows are mapped by the reduction
      const int orow = row >= Mdev ? -1
                       : (direct && p.row_map != nullptr) ? __ldg(p.row_map + row) : row;
      const uint32_t t_acc =
          tmem + static_cast<uint32_t>(a * p.acc_cols) + (static_cast<uint32_t>(q * 32) << 16);
      for (int c = 0; c < w.bn; c += 16) {
        uint32_t v[16];
        tmem_ld16(t_acc + c, v);
        if (orow >= 0) {
          float4* dst =
              reinterpret_cast<float4*>(dst_base + static_cast<size_t>(orow) * p.d + w.n0 + c);
          if (w.nkb == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0u;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                 __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(acce0 + 8 * a, 0));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_v) {
    // drain (bounded): MMAs already issued must finish, and TMA boxes still in flight must
    // land, before shared memory and TMEM go away.  Both CTAs' boxes complete on the leader's
    // barriers, and the peer waits at the cluster barrier below until the leader has drained.
    if (leader && last_k >= 0 && lane == 0) drain_bar(full0 + 8 * (last_k % S), (last_k / S) & 1);
    __syncthreads();
  }
  // every MMA has completed (in both CTAs: the commit is multicast) before TMEM is freed
  if (warp == 0 && lane == 0) drain_bar(done_bar, 0);
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or signals may still touch it
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, p.tmem_cols);
  }
}

__global__ void splitk_reduce_kernel(const float* part, int split_k, int R_pad, int d,
                                     const int32_t* M, const int32_t* row_map, float* out) {
  pdl_wait();
  const int Mdev = *M;
  const int d4 = d / 4;
  const size_t n4 = static_cast<size_t>(Mdev) * d4;
  const size_t slice = static_cast<size_t>(R_pad) * d4;
  const float4* p4 = reinterpret_cast<const float4*>(part);
  float4* o4 = reinterpret_cast<float4*>(out);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(i / d4);
    const int orow = row_map != nullptr ? __ldg(row_map + row) : row;
    if (orow < 0) continue;
    float4 acc = p4[i];
    for (int k = 1; k < split_k; ++k) {  // fixed order: deterministic
      const float4 v = p4[k * slice + i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    o4[static_cast<size_t>(orow) * d4 + (i - static_cast<size_t>(row) * d4)] = acc;
  }
}

// ------------------------------------------------------------------ probability rows

constexpr int kProbThreads = 256;

// P[j, v] = bf16_rn(exp(z_{r_j, v} - lse_{r_j})) for j < M, 8 elements per thread-step, stored
// K-slab-blocked: element (j, v) at ((v / 64) * R_pad + j) * 64 + v % 64.  The columns of the
// last slab beyond V are written as zeros (the GEMM reads whole slabs).  kScalar: rows that are
// not 16-byte aligned (an odd row stride, an element-aligned pointer) or V not a multiple of 8
// are read element by element.
template <int DT, bool kScalar>
__global__ void __launch_bounds__(kProbThreads) prob_rows_kernel(const char* logits,
                                                                 int64_t row_stride_bytes, int V,
                                                                 int S, int chunk,
                                                                 const float* lse,
                                                                 const int32_t* row_ids,
                                                                 const int32_t* M, uint16_t* P,
                                                                 int R_pad) {
  const int j = blockIdx.x / S;
  const int split = blockIdx.x - j * S;
  pdl_wait();
  pdl_trigger();
  if (j >= *M) return;
  const int r = row_ids[j];
  const float mb = lse[r] * kLog2e;
  const char* row = logits + static_cast<int64_t>(r) * row_stride_bytes;
  const int e0 = split * chunk;
  const int e1 = min(static_cast<int>(align_up(V, 64)), e0 + chunk);
  const int ngroups = (e1 - e0) / 8;
  for (int g = threadIdx.x; g < ngroups; g += kProbThreads) {
    const int e = e0 + g * 8;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (e < V) {
      float x[8];
      if constexpr (kScalar) {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = e + k < V ? load_logit(row, DT, e + k) : -INFINITY;
      } else if constexpr (DT == DLLM_BF16) {
        unpack_vec<DT>(ld_stream_v4(row + static_cast<int64_t>(e) * 2), x);
      } else {
        unpack_vec<DT>(ld_stream_v4(row + static_cast<int64_t>(e) * 4), x);
        unpack_vec<DT>(ld_stream_v4(row + static_cast<int64_t>(e) * 4 + 16), x + 4);
      }
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float lo = ex2(fmaf(x[2 * h], kLog2e, -mb));
        const float hi = ex2(fmaf(x[2 * h + 1], kLog2e, -mb));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[h]) : "f"(hi), "f"(lo));
      }
      out = make_uint4(w[0], w[1], w[2], w[3]);
    }
    uint16_t* dst = P + ((static_cast<int64_t>(e >> 6) * R_pad + j) << 6) + (e & 63);
    *reinterpret_cast<uint4*>(dst) = out;
  }
}

// ------------------------------------------------------------------ embedding relayout

constexpr int kTT = 32;

// Et[(v / 64) * d + c][v % 64] = E[v][c]  (K-slab-blocked transpose; zeros for v >= V).
__global__ void transpose_bf16_kernel(const uint16_t* E, int V, int d, uint16_t* Et, int Vp) {
  __shared__ uint16_t tile[kTT][kTT + 2];
  const int v0 = blockIdx.x * kTT, c0 = blockIdx.y * kTT;
  for (int y = threadIdx.y; y < kTT; y += blockDim.y) {
    const int v = v0 + y, c = c0 + threadIdx.x;
    tile[y][threadIdx.x] = (v < V && c < d) ? E[static_cast<int64_t>(v) * d + c] : uint16_t(0);
  }
  __syncthreads();
  for (int y = threadIdx.y; y < kTT; y += blockDim.y) {
    const int c = c0 + y, v = v0 + threadIdx.x;
    if (c < d && v < Vp)
      Et[((static_cast<int64_t>(v >> 6) * d + c) << 6) + (v & 63)] = tile[threadIdx.x][y];
  }
}

// ------------------------------------------------------------------ host side

constexpr size_t kMaxDynSmem = 227 * 1024;

}  // namespace

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no libcuda link).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// K-slab-blocked bf16 operand [slabs][rows][64] as a 3-D tensor map; boxes of
// 64 x box_rows x box_slabs with 128-byte swizzle (the K-major layout the tcgen05 descriptors
// expect; the slabs of a box land one after another in shared memory).  Rows or slabs of a box
// beyond the tensor read as zeros.
bool make_slab_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t slabs,
                   uint32_t box_rows, uint32_t box_slabs) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, slabs};
  cuuint64_t strides[2] = {128, rows * 128};
  cuuint32_t box[3] = {64, box_rows, box_slabs};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

SmoothPlan smooth_plan(int B, int L, int V, int d, int sm_count) {
  SmoothPlan pl{};
  pl.R = B * L;
  pl.V = V;
  pl.d = d;
  pl.ldp = static_cast<int>(align_up(V, 64));  // slabs x 64
  const int m_pairs = (pl.R + 2 * kBM - 1) / (2 * kBM);
  pl.m_tiles = 2 * m_pairs;
  const int units16 = d / 16;
  const int num_kb = (V + kBK - 1) / kBK;
  const int pair_slots = std::max(1, sm_count / 2);
  // Pick (column tiles, split-K, tail pairs) for one wave of CTA pairs, minimising the K blocks
  // of the busiest pair x (BN + 64): wide tiles carry more MMA work per byte staged, and each
  // extra K range costs a round trip of fp32 partial sums.  Pair slots that the main pairs
  // (every tile over split-K equal ranges) leave free take tail pairs: the main ranges stop
  // short of V and each tail pair runs a few tiles over the remaining K blocks, so that every
  // pair streams about as many K blocks and no SM idles.  Only when one wave cannot hold the
  // grid are more waves allowed (then each wave is charged in full).
  double best = 1e300;
  for (int nt = (units16 + 15) / 16; nt <= units16; ++nt) {
    const int base = units16 / nt, rem = units16 % nt;
    const int bn_max = (base + (rem ? 1 : 0)) * 16;
    if (bn_max > 256) continue;
    const size_t slab_b = kATileBytes + static_cast<size_t>(bn_max / 2) * kBK * 2;
    const int G = (kMaxDynSmem - 2048) / (2 * slab_b) >= 3 ? 2 : 1;  // slabs per stage
    const int tiles = m_pairs * nt;
    for (int sk = 1; sk <= std::min(8, num_kb); ++sk) {
      const long pairs = static_cast<long>(tiles) * sk;
      const long waves = (pairs + pair_slots - 1) / pair_slots;
      const int kbs = (num_kb + sk - 1) / sk;
      const double split_cost = 0.02 * num_kb * 256.0;
      double est = (waves > 1 ? 4.0 * waves : 1.0) * kbs * (bn_max + 64.0) +
                   (sk > 1 ? split_cost * sk : 0.0);
      int tp = 0, tt = 0, km = kbs;
      const int free_slots = pair_slots - static_cast<int>(pairs);
      if (waves == 1 && free_slots > 0 && G == 2) {
        // tail pairs: tt consecutive column tiles of one row pair each, tt dividing the column
        // tiles (so the tail pairs running at one time read the same few column tiles of E^T,
        // each shared by every row pair, and a pair keeps its P rows); main ranges of km
        // blocks (a whole number of stages)
        int t_tt = 1;
        while (t_tt <= nt && (nt % t_tt != 0 || tiles / t_tt > free_slots)) ++t_tt;
        if (t_tt > nt) t_tt = 0;
        const int t_tp = t_tt > 0 ? tiles / t_tt : 0;
        int t_km = t_tt > 0
                       ? static_cast<int>(static_cast<double>(num_kb) * t_tt / (sk * t_tt + 1))
                       : 0;
        t_km -= t_km % G;
        if (t_tt > 0 && t_km >= 8 * G && sk * t_km < num_kb) {
          const int tail = num_kb - sk * t_km;
          const double work = std::max(t_km, t_tt * tail + 2 * (t_tt - 1));
          const double t_est = work * (bn_max + 64.0) + split_cost * (sk + 1);
          if (t_est < est) {
            est = t_est;
            tp = t_tp;
            tt = t_tt;
            km = t_km;
          }
        }
      }
      if (est < best - 1e-9) {
        best = est;
        pl.n_tiles = nt;
        pl.bn_max = bn_max;
        pl.split_k = sk;
        pl.kb_per_split = km;
        pl.tail_pairs = tp;
        pl.tail_tiles = tt;
        pl.kb_tail0 = tp > 0 ? sk * km : num_kb;
      }
    }
  }
  pl.partials = pl.split_k + (pl.tail_pairs > 0 ? 1 : 0);
  // Two slabs per stage halve the stage hand-offs per MMA (three stages fit); one slab when
  // two would leave fewer than three stages.
  const size_t slab_bytes = kATileBytes + static_cast<size_t>(pl.bn_max / 2) * kBK * 2;
  pl.slabs_per_stage = (kMaxDynSmem - 2048) / (2 * slab_bytes) >= 3 ? 2 : 1;
  const size_t stage_bytes = pl.slabs_per_stage * slab_bytes;
  pl.stages = static_cast<int>(std::min<size_t>(kMaxStages, (kMaxDynSmem - 2048) / stage_bytes));
  pl.stages = std::min(pl.stages, kProducers);  // one producer warp per stage
  const int R_pad = pl.m_tiles * kBM;
  size_t off = kWsHeader;
  off = align_up(off, 1024);
  pl.off_p = off;
  off += static_cast<size_t>(R_pad) * pl.ldp * 2;
  off = align_up(off, 1024);
  pl.off_part = off;
  if (pl.partials > 1) off += static_cast<size_t>(pl.partials) * R_pad * d * 4;
  const size_t rows4 = align_up(4 * static_cast<size_t>(pl.R), 256);
  off = align_up(off, 256);
  pl.off_rows = off;
  off += rows4;
  pl.off_count = off;
  off += 256;
  pl.off_inv = off;
  off += rows4;
  pl.off_map = off;
  off += rows4;
  off = align_up(off, 256);
  pl.off_stats_ws = off;
  off += stats_ws_bytes(B, L, V);
  pl.ws_bytes = align_up(off, 256);
  return pl;
}

cudaError_t launch_prob_rows(const void* logits, const dllm_shape& sh, const float* lse,
                             const int32_t* row_ids, const int32_t* M, uint16_t* P, int R_pad,
                             int sm_count, cudaStream_t stream) {
  const int R = sh.B * sh.L;
  const int es = sh.dtype == DLLM_BF16 ? 2 : 4;
  // ~32 KB of logits per CTA, at least ~8 CTAs per SM
  int S = std::max(1, sh.V / (32768 / es));
  while (static_cast<int64_t>(R) * S < static_cast<int64_t>(sm_count) * 8 && sh.V / (S * 2) >= 2048)
    S *= 2;
  const int Vp = static_cast<int>(align_up(sh.V, 64));
  int chunk = static_cast<int>(align_up((Vp + S - 1) / S, 8));
  S = (Vp + chunk - 1) / chunk;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(R) * S));
  const int64_t rsb = sh.row_stride * es;
  const char* lg = static_cast<const char*>(logits);
  const bool scalar = reinterpret_cast<uintptr_t>(logits) % 16 != 0 || rsb % 16 != 0 ||
                      sh.V % 8 != 0;
  auto kern = sh.dtype == DLLM_BF16
                  ? (scalar ? prob_rows_kernel<DLLM_BF16, true> : prob_rows_kernel<DLLM_BF16, false>)
                  : (scalar ? prob_rows_kernel<DLLM_F32, true> : prob_rows_kernel<DLLM_F32, false>);
  return launch_dependent(kern, grid, dim3(kProbThreads), 0, stream, lg, rsb, sh.V, S, chunk, lse,
                          row_ids, M, P, R_pad);
}

cudaError_t launch_smooth_gemm(const SmoothPlan& pl, const uint16_t* P, const uint16_t* Et,
                               int ldt, float* out, const int32_t* M, const int32_t* row_map,
                               bool wait_late, void* ws, cudaStream_t stream, const char** why) {
  const int R_pad = pl.m_tiles * kBM;
  (void)ldt;
  GemmParams gp{};
  const uint64_t slabs = static_cast<uint64_t>(pl.ldp) / 64;
  const int G = std::max(1, pl.slabs_per_stage);
  if (!make_slab_map(&gp.tmA, P, R_pad, slabs, kBM, G) ||
      !make_slab_map(&gp.tmB, Et, pl.d, slabs, pl.bn_max / 2, G)) {
    *why = "cuTensorMapEncodeTiled failed or is unavailable (E^T must be 16-byte aligned)";
    return cudaErrorInvalidValue;
  }
  gp.num_kb = (pl.V + kBK - 1) / kBK;
  gp.n_tiles = pl.n_tiles;
  const int units16 = pl.d / 16;
  gp.bn_base = (units16 / pl.n_tiles) * 16;
  gp.bn_rem = units16 % pl.n_tiles;
  gp.bn_max = pl.bn_max;
  gp.split_k = pl.split_k;
  gp.kb_per_split = pl.kb_per_split;
  gp.main_pairs = pl.m_tiles / 2 * pl.n_tiles * pl.split_k;
  gp.tail_pairs = pl.tail_pairs;
  gp.tail_tiles = pl.tail_tiles;
  gp.kb_tail0 = pl.kb_tail0;
  gp.stages = pl.stages;
  gp.gs = G;
  if (pl.tail_pairs > 0) {  // two accumulators of up to 256 columns: the whole tensor memory
    gp.tmem_cols = 512;
    gp.acc_cols = 256;
  } else {
    int cols = 32;
    while (cols < pl.bn_max) cols *= 2;
    gp.tmem_cols = cols;
    gp.acc_cols = 0;
  }
  gp.d = pl.d;
  gp.R_pad = R_pad;
  gp.out = out;
  gp.part = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_part);
  gp.M = M;
  gp.row_map = row_map;
  gp.status = static_cast<int32_t*>(ws);
  gp.wait_late = wait_late ? 1 : 0;
  const size_t smem = static_cast<size_t>(pl.stages) * G *
                          (kATileBytes + static_cast<size_t>(pl.bn_max / 2) * kBK * 2) + 1024;
  cudaError_t e = cudaFuncSetAttribute(smooth_gemm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // two CTAs (a cluster) per main or tail pair
  const dim3 grid(static_cast<unsigned>(2 * (gp.main_pairs + gp.tail_pairs)));
  e = launch_dependent(smooth_gemm_kernel, grid, dim3(kGemmThreads), smem, stream, gp);
  if (e != cudaSuccess || pl.partials == 1) return e;
  return launch_dependent(splitk_reduce_kernel,
                          dim3(std::min(1024, std::max(1, pl.R * pl.d / 4 / 256))), dim3(256), 0,
                          stream, static_cast<const float*>(gp.part), pl.partials, R_pad, pl.d, M,
                          row_map, out);
}

cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_transpose_embedding(const uint16_t* E, int V, int d, uint16_t* Et, int Vp,
                                       cudaStream_t stream) {
  const dim3 grid((Vp + kTT - 1) / kTT, (d + kTT - 1) / kTT);
  transpose_bf16_kernel<<<grid, dim3(kTT, 8), 0, stream>>>(E, V, d, Et, Vp);
  return cudaGetLastError();
}

}  // namespace dllm
