// bf16 cross-entropy on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent, warp-specialised kernel template serves the four
// contractions of the loss ("Vocabulary shards: look up locally and normalize
// globally", paragraphs 3-5):
//   FWD   z = h W^T per (256-token block, work unit inside one shard): the
//         epilogue keeps a running maximum and sum of exp per token over the
//         unit's real columns (padded classes >= V_real never count) and picks
//         the target logit from the one tile that owns it. Logits stay in TMEM.
//   GRAD  z recomputed per 256 x 256 tile; the epilogue forms
//         G = (exp(z - lse) - [v == y]) * g / N_valid in bf16 and stores it.
//   DH    dH (+)= G W      (A = G K-major, B = W rows as an MN-major operand)
//   DW    dW (+)= G^T h    (A = G^T and B = h, both MN-major operands)
//
// Two CTAs on two SMs form a cluster and share each MMA (tcgen05 cta_group::2,
// M = 256, N = 256, K = 16): each CTA loads 128 rows of A and half of B's N
// range into its own shared memory, and each CTA's TMEM receives its 128 rows
// of the 256 x 256 fp32 tile. Per SM this halves the B traffic through shared
// memory compared with a 128 x 256 single-SM tile.
//
// Roles (320 threads per CTA): warp 0 issues TMA loads into a ring of stages;
// their completion is counted on the even CTA's barrier. Warp 1 allocates 512
// TMEM columns (two accumulators) in both CTAs; in the even CTA one lane issues
// the MMAs and commits to the barriers of both CTAs. Warps 2-9 of both CTAs
// drain their own TMEM (warp w reads lanes 32*(w%4)..+31, one token row per
// thread, and one 128-column half of the tile) with software-pipelined TMEM
// loads, and release the accumulator to the even CTA. Every wait is bounded:
// on a timeout the CTA raises its abort flag, records VCE_ERR_TIMEOUT, drains
// what it has in flight and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace vce {
namespace {

constexpr int BM = 128;          // A rows per CTA
constexpr int BMP = 256;         // A rows per CTA pair (the MMA's M)
constexpr int BN = 256;          // the MMA's N (tile columns)
constexpr int BNH = 128;         // N rows of B held by each CTA
constexpr int BK = 64;
constexpr int kEpiWarps = 8;                   // two per TMEM lane quarter, one per 128-column half
constexpr int kThreads = 64 + 32 * kEpiWarps;   // producer warp, MMA warp, epilogue warps
constexpr uint32_t kABytes = BM * BK * 2;    // 16 KB
constexpr uint32_t kBBytes = BNH * BK * 2;   // 16 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kAtomBytes = 64 * 128;        // 64 rows of 128 B: one MN-major atom column
constexpr uint32_t kStagingPerWarp = 4096;       // one 32-row x 128-B TMA store box
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

enum Mode : int { MODE_FWD = 0, MODE_GRAD = 1, MODE_DH = 2, MODE_DW = 3, MODE_ARGMAX = 4 };
// FWD and ARGMAX share the logit GEMM and its work items; they differ in the epilogue.
template <int MODE>
constexpr bool kFwdLike = MODE == MODE_FWD || MODE == MODE_ARGMAX;

template <int MODE>
struct Traits {
  static constexpr uint32_t a_mn = (MODE == MODE_DW) ? 1u : 0u;
  static constexpr uint32_t b_mn = (MODE == MODE_DH || MODE == MODE_DW) ? 1u : 0u;
  static constexpr bool staging = !kFwdLike<MODE>;
  static constexpr int stages = 6;
  static constexpr uint32_t idesc = idesc_bf16_f32(BMP, BN, a_mn, b_mn);
};

template <int MODE>
constexpr size_t smem_bytes() {
  return 1024 + size_t(Traits<MODE>::stages) * kStageBytes +
         (Traits<MODE>::staging ? kEpiWarps * kStagingPerWarp : 0) + 256 + (kFwdLike<MODE> ? 2048 : 0);
}

struct TcArgs {
  ProbDev pd;
  const int64_t* targets;
  int n_items;
  int n_mblk;
  int n_nblk;
  int num_kb;
  UnitGrid ug;
  float2* part;
  float* ztgt;
  const float* lse;
  float g;
  int v0;
  int vc;
  int out_row0;
  int accumulate;
  int ksplit;    // DH: the K range (vocabulary columns) is cut into ksplit parts
  int kb_per;    // DH: K blocks per part
  int32_t* dh_flags;   // DH with ksplit > 1: per (tile, CTA, epilogue warp), parts added so far;
                       // GRAD zeroes them for the DH launch that follows it
  int n_dh_flags;
  int gm;        // FWD, ARGMAX, GRAD: token blocks per item group (see item_mc)
  int n_cols;    // FWD, ARGMAX: units; GRAD: column blocks
  int32_t* status;
  uint64_t limit_ns;
  int32_t* merge_ctr;   // FWD: the merge's block counter, zeroed here for the merge that follows
};

// Items of the forward-like modes and of GRAD are (token block m, column
// unit or block c) pairs, taken in groups of gm token blocks: group g covers
// m in [g*gm, g*gm + gsz) and every c, c-major within the group. The clusters
// working at the same time then share one or two column blocks and at most gm
// blocks of h, a working set chosen to stay in L2 (with gm = n_mblk this is
// plain c-major order).
struct MC {
  int m, c;
};
__host__ __device__ __forceinline__ MC item_mc(int item, int gm, int n_mblk, int n_cols) {
  const int per_group = gm * n_cols;
  const int g = item / per_group, r = item - g * per_group;
  const int m0 = g * gm;
  const int gsz = n_mblk - m0 < gm ? n_mblk - m0 : gm;
  return MC{m0 + r % gsz, r / gsz};
}

// Columns [vb, vlim) of forward work unit u, and its number of 256-wide tiles.
struct UnitSpan {
  int64_t vb, vlim;
  int ntiles;
};
__device__ __forceinline__ UnitSpan unit_span(const TcArgs& a, int u) {
  const int k = u / a.ug.ups, j = u - k * a.ug.ups;
  const int64_t lo = shard_lo(k, a.pd.Vp, a.pd.S), hi = shard_lo(k + 1, a.pd.Vp, a.pd.S);
  UnitSpan s;
  s.vb = lo + static_cast<int64_t>(j) * a.ug.uw;
  int64_t ve = s.vb + a.ug.uw;
  if (ve > hi) ve = hi;
  s.vlim = ve < a.pd.V_real ? ve : a.pd.V_real;
  s.ntiles = s.vlim > s.vb ? static_cast<int>((s.vlim - s.vb + BN - 1) / BN) : 0;
  return s;
}

template <int MODE>
__device__ __forceinline__ int item_tiles(const TcArgs& a, int item) {
  if constexpr (kFwdLike<MODE>) {
    return unit_span(a, item_mc(item, a.gm, a.n_mblk, a.n_cols).c).ntiles;
  } else {
    return 1;
  }
}

// This CTA's tile origin: am = first of its 128 rows of A's M range, bn =
// first of its 128 indices of B's N range (a vocabulary row for FWD/GRAD, an
// H column for DH/DW). Computed once per tile.
struct TileCoord {
  int32_t am, bn;
};
template <int MODE>
__device__ __forceinline__ TileCoord tile_coord(const TcArgs& a, int item, int tt, int rank) {
  TileCoord c;
  if constexpr (kFwdLike<MODE>) {
    const MC mc = item_mc(item, a.gm, a.n_mblk, a.n_cols);
    const UnitSpan us = unit_span(a, mc.c);
    c.am = mc.m * BMP + rank * BM;
    c.bn = static_cast<int32_t>(us.vb + static_cast<int64_t>(tt) * BN) + rank * BNH;
  } else if constexpr (MODE == MODE_GRAD) {
    const MC mc = item_mc(item, a.gm, a.n_mblk, a.n_cols);
    c.am = mc.m * BMP + rank * BM;
    c.bn = a.v0 + mc.c * BN + rank * BNH;
  } else {
    const int n_blk = item % a.n_nblk, m_blk = (item / a.n_nblk) % a.n_mblk;
    c.am = m_blk * BMP + rank * BM;
    c.bn = n_blk * BN + rank * BNH;
  }
  return c;
}

// K blocks [kb0, kb1) of an item: all of K, except for DH cut into parts.
// DH and DW items are (part * n_mblk + m_blk) * n_nblk + n_blk: the parts run
// one after the other, so the clusters working at the same time read one K
// range of W.
struct KRange {
  int kb0, kb1;
};
template <int MODE>
__device__ __forceinline__ KRange item_krange(const TcArgs& a, int item) {
  if constexpr (MODE == MODE_DH) {
    const int part = (item / a.n_nblk) / a.n_mblk;
    const int kb0 = part * a.kb_per;
    const int kb1 = kb0 + a.kb_per < a.num_kb ? kb0 + a.kb_per : a.num_kb;
    return KRange{kb0, kb1};
  } else {
    return KRange{0, a.num_kb};
  }
}

template <int MODE>
__device__ __forceinline__ void issue_loads(const TcArgs& a, const CUtensorMap* mA, const CUtensorMap* mB,
                                            uint32_t sA, uint32_t sB, uint32_t bar, TileCoord c, int kb) {
  const int k0 = kb * BK;
  if constexpr (kFwdLike<MODE> || MODE == MODE_GRAD) {
    tma_load_2d_pair(sA, mA, bar, k0, c.am);
    tma_load_2d_pair(sB, mB, bar, k0, c.bn);
  } else if constexpr (MODE == MODE_DH) {
    tma_load_2d_pair(sA, mA, bar, k0, c.am);
#pragma unroll
    for (int b = 0; b < 2; ++b) tma_load_2d_pair(sB + b * kAtomBytes, mB, bar, c.bn + 64 * b, a.v0 + k0);
  } else {
#pragma unroll
    for (int b = 0; b < 2; ++b) tma_load_2d_pair(sA + b * kAtomBytes, mA, bar, c.am + 64 * b, k0);
#pragma unroll
    for (int b = 0; b < 2; ++b) tma_load_2d_pair(sB + b * kAtomBytes, mB, bar, c.bn + 64 * b, k0);
  }
}

__device__ __forceinline__ float select32(const uint32_t (&x)[32], int idx) {
  float r = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (j == idx) r = __uint_as_float(x[j]);
  return r;
}

// Writes one thread's 128-byte row into a 32-row staging box laid out with
// the 128-byte swizzle a TMA store expects (16-byte chunk c of row r at
// c ^ (r % 8)).
__device__ __forceinline__ void stage_row(uint32_t box, int r, const uint32_t (&w)[32]) {
  const uint32_t row = box + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t addr = row + ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(r & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * c]), "r"(w[4 * c + 1]),
                 "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                 : "memory");
  }
}

__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_loss_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapOut, const TcArgs a) {
  using Tr = Traits<MODE>;
  constexpr int kStages = Tr::stages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t stage0 = base;
  const uint32_t staging0 = base + kStages * kStageBytes;
  uint8_t* tail = gbase + kStages * kStageBytes + (Tr::staging ? kEpiWarps * kStagingPerWarp : 0);
  uint64_t* full = reinterpret_cast<uint64_t*>(tail);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* comb_full = drain + 1;     // forward: half-row partial handoff per lane quarter
  uint64_t* comb_empty = comb_full + 4;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(comb_empty + 4);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);
  int* s_cnt = reinterpret_cast<int*>(tail + 216);   // GRAD: the epilogue warps' valid-target counts
  float4* comb = reinterpret_cast<float4*>(tail + 256);   // [4 quarters][32 lanes], forward only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int first_item = static_cast<int>(cluster_id_x());
  const int item_step = static_cast<int>(cluster_count_x());
  grid_dep_launch();   // the next kernel may set itself up once every CTA is here
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);     // the even CTA's expect_tx; bytes from both CTAs
      mbar_init(&empty[s], 1);    // one multicast commit per use
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 2 * kEpiWarps);   // every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&comb_full[s], 1);
      mbar_init(&comb_empty[s], 1);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const WaitCtx wc{s_abort, a.status, a.limit_ns};
  // Launched as a dependent launch: barriers and TMEM are set up while the
  // previous kernel drains; nothing in global memory is touched before it ends.
  grid_dep_wait();
  if constexpr (MODE == MODE_FWD) {
    if (a.merge_ctr && blockIdx.x == 0 && threadIdx.x == 0) *a.merge_ctr = 0;
  }
  if constexpr (MODE == MODE_GRAD) {   // the next DH launch's part counters start at zero
    for (int i = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x); i < a.n_dh_flags;
         i += static_cast<int>(gridDim.x * blockDim.x))
      a.dh_flags[i] = 0;
  }

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB);
      int stage = 0;
      uint32_t phase = 0;
      // the even CTA's full barriers, as cluster addresses (consecutive words)
      const uint32_t full_leader0 = mapa_shared(smem_u32(&full[0]), 0);
      int last_parity[kStages];
#pragma unroll
      for (int s = 0; s < kStages; ++s) last_parity[s] = -1;
      bool ok = true, issued = false;
      for (int item = first_item; ok && item < a.n_items; item += item_step) {
        const int nt = item_tiles<MODE>(a, item);
        for (int tt = 0; ok && tt < nt; ++tt) {
          const TileCoord tc = tile_coord<MODE>(a, item, tt, static_cast<int>(rank));
          const KRange kr = item_krange<MODE>(a, item);
          for (int kb = kr.kb0; kb < kr.kb1; ++kb) {
            if (!mbar_wait_cl(&empty[stage], phase ^ 1u, wc)) {
              ok = false;
              break;
            }
            const uint32_t full_leader = full_leader0 + static_cast<uint32_t>(stage) * 8u;
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
            const uint32_t sA = stage0 + stage * kStageBytes;
            issue_loads<MODE>(a, &mapA, &mapB, sA, sA + kABytes, full_leader, tc, kb);
            issued = true;
            last_parity[stage] = static_cast<int>(phase);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && issued) {
        // Let the copies already issued land before the CTA's memory goes away.
        const uint64_t t0 = globaltimer_ns();
        if (leader) {
          for (int s = 0; s < kStages; ++s) {
            if (last_parity[s] < 0) continue;
            while (!mbar_try_wait_cluster(&full[s], static_cast<uint32_t>(last_parity[s])) &&
                   globaltimer_ns() - t0 < 100000000ull) {
            }
          }
        } else {
          while (globaltimer_ns() - t0 < 2000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (even CTA) ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tile_count = 0;
      bool ok = true;
      bool issued = false;
      for (int item = first_item; ok && item < a.n_items; item += item_step) {
        const int nt = item_tiles<MODE>(a, item);
        for (int tt = 0; ok && tt < nt; ++tt) {
          const uint32_t acc = tile_count & 1u;
          if (!mbar_wait_cl(&tempty[acc], ((tile_count >> 1) & 1u) ^ 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + acc * BN;
          const KRange kr = item_krange<MODE>(a, item);
          for (int kb = kr.kb0; kb < kr.kb1; ++kb) {
            if (!mbar_wait_cl(&full[stage], phase, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sA = stage0 + stage * kStageBytes;
            const uint32_t sB = sA + kABytes;
            const uint64_t ad0 = Tr::a_mn ? smem_desc_sw128(sA, kAtomBytes, 1024u) : smem_desc_sw128(sA, 16u, 1024u);
            const uint64_t bd0 = Tr::b_mn ? smem_desc_sw128(sB, kAtomBytes, 1024u) : smem_desc_sw128(sB, 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = ad0 + static_cast<uint64_t>(Tr::a_mn ? kk * (2048u >> 4) : kk * (32u >> 4));
              const uint64_t bd = bd0 + static_cast<uint64_t>(Tr::b_mn ? kk * (2048u >> 4) : kk * (32u >> 4));
              umma_f16_pair(d, ad, bd, Tr::idesc, (kb != kr.kb0 || kk != 0) ? 1u : 0u);
            }
            issued = true;
            umma_commit_pair_mc(&empty[stage], 0x3);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair_mc(&tfull[acc], 0x3);
          ++tile_count;
        }
      }
      if (!ok && issued) {
        // Wait for the MMAs in flight before TMEM is released.
        umma_commit_pair(drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 2..9 of both CTAs ----------------
    // Warps e and e+4 (e = warp - 2) share TMEM lane quarter warp % 4; warp e
    // takes tile columns [128 * (e / 4), +128).
    const int e = warp - 2;
    const int q = warp & 3;
    const int half = e >> 2;
    const int pq = e & 3;
    const int r = q * 32 + lane;      // row of this CTA's half tile held by this thread
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(half * 128);
    const uint32_t my_staging = staging0 + static_cast<uint32_t>(e) * kStagingPerWarp;
    const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty[1]), 0);
    uint32_t tile_count = 0;
    uint32_t items_done = 0;
    bool ok = true;
    float scale = 0.0f;
    if constexpr (MODE == MODE_GRAD) {
      // N_valid, the mean's denominator: the epilogue warps of every CTA count
      // the valid targets themselves (T int64 reads from L2) while the first
      // tile's MMAs run, so no separate counting launch precedes the backward.
      int cnt = 0;
      bool bad = false;
      constexpr int kStep = 32 * kEpiWarps;
      // eight independent loads in flight per thread, then their tests
      for (int t0 = static_cast<int>(threadIdx.x) - 64; t0 < a.pd.T; t0 += 8 * kStep) {
        int64_t y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = t0 + j * kStep < a.pd.T ? __ldg(a.targets + t0 + j * kStep) : a.pd.ignore_index;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool v = (y[j] >= 0) && (y[j] < a.pd.V_real);
          cnt += v ? 1 : 0;
          bad |= !v && y[j] != a.pd.ignore_index;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) s_cnt[e] = cnt;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");   // the epilogue warps only
      int nv = 0;
#pragma unroll
      for (int w = 0; w < kEpiWarps; ++w) nv += s_cnt[w];
      if (bad && lane == 0 && blockIdx.x == 0) record_status(a.status, VCE_ERR_BAD_INDEX);
      scale = nv > 0 ? a.g / static_cast<float>(nv) : 0.0f;
    }
    auto release = [&](uint32_t acc) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
    };
    // One 32-row x 128-byte TMA store (or reduce-add) from this warp's staging box.
    bool add_out = MODE != MODE_GRAD && a.accumulate;
    auto store_box = [&](const uint32_t (&w)[32], int col, int row) {
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      stage_row(my_staging, lane, w);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (add_out)
          tma_reduce_add_2d(&mapOut, my_staging, col, row);
        else
          tma_store_2d(&mapOut, my_staging, col, row);
        bulk_commit();
      }
    };
    for (int item = first_item; ok && item < a.n_items; item += item_step) {
      if constexpr (MODE == MODE_ARGMAX) {
        const MC mc = item_mc(item, a.gm, a.n_mblk, a.n_cols);
        const int m_blk = mc.m, u = mc.c;
        const UnitSpan us = unit_span(a, u);
        const int t = m_blk * BMP + static_cast<int>(rank) * BM + r;
        float m_run = -INFINITY;
        int32_t i_run = -1;
        // Largest real logit of one 32-column chunk; strict > keeps the lowest column.
        auto chunk = [&](const uint32_t (&x)[32], int64_t vc0) {
          const int64_t nval64 = us.vlim - vc0;
          const int nval = nval64 >= 32 ? 32 : (nval64 <= 0 ? 0 : static_cast<int>(nval64));
          float best = -INFINITY;
          int bj = -1;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float v = __uint_as_float(x[j]);
            if (j < nval && v > best) {
              best = v;
              bj = j;
            }
          }
          if (bj >= 0 && best > m_run) {
            m_run = best;
            i_run = static_cast<int32_t>(vc0) + bj;
          }
        };
        for (int tt = 0; tt < us.ntiles; ++tt) {
          const uint32_t acc = tile_count & 1u;
          if (!mbar_wait_cl(&tfull[acc], (tile_count >> 1) & 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int64_t vc = us.vb + static_cast<int64_t>(tt) * BN + half * 128;
          const uint32_t ta = lane_base + acc * BN;
          uint32_t xa[32], xb[32];
          tmem_ld_32x32b_x32(ta, xa);
          tmem_ld_wait();
          reg_fence(xa);
          tmem_ld_32x32b_x32(ta + 32, xb);
          chunk(xa, vc);
          tmem_ld_wait();
          reg_fence(xb);
          tmem_ld_32x32b_x32(ta + 64, xa);
          chunk(xb, vc + 32);
          tmem_ld_wait();
          reg_fence(xa);
          tmem_ld_32x32b_x32(ta + 96, xb);
          chunk(xa, vc + 64);
          tmem_ld_wait();
          reg_fence(xb);
          release(acc);
          chunk(xb, vc + 96);
          ++tile_count;
        }
        if (!ok) break;
        // Join the two column halves: the larger logit, the lower column on a tie.
        if (half == 1) {
          if (!mbar_wait(&comb_empty[pq], (items_done & 1u) ^ 1u, wc)) {
            ok = false;
            break;
          }
          comb[pq * 32 + lane] = make_float4(m_run, __int_as_float(i_run), 0.0f, 0.0f);
          __syncwarp();
          if (lane == 0) mbar_arrive(&comb_full[pq]);
        } else {
          if (!mbar_wait(&comb_full[pq], items_done & 1u, wc)) {
            ok = false;
            break;
          }
          const float4 o = comb[pq * 32 + lane];
          __syncwarp();
          if (lane == 0) mbar_arrive(&comb_empty[pq]);
          const int32_t oi = __float_as_int(o.y);
          if (oi >= 0 && (i_run < 0 || o.x > m_run || (o.x == m_run && oi < i_run))) {
            m_run = o.x;
            i_run = oi;
          }
          if (t < a.pd.T) a.part[static_cast<int64_t>(t) * a.ug.n_units + u] = make_float2(m_run, __int_as_float(i_run));
        }
        ++items_done;
      } else if constexpr (MODE == MODE_FWD) {
        const MC mc = item_mc(item, a.gm, a.n_mblk, a.n_cols);
        const int m_blk = mc.m, u = mc.c;
        const UnitSpan us = unit_span(a, u);
        const int t = m_blk * BMP + static_cast<int>(rank) * BM + r;
        const bool row_ok = t < a.pd.T;
        const int64_t y = row_ok ? a.targets[t] : -1;
        float m_run = -INFINITY, s_run = 0.0f, zt = 0.0f;
        bool have_zt = false;
        // Online maximum and sum of exp over one 32-column chunk of real columns.
        auto chunk = [&](const uint32_t (&x)[32], int64_t vc0) {
          const int64_t nval64 = us.vlim - vc0;
          const int nval = nval64 >= 32 ? 32 : (nval64 <= 0 ? 0 : static_cast<int>(nval64));
          if (nval == 0) return;
          if (y >= vc0 && y < vc0 + nval) {
            zt = select32(x, static_cast<int>(y - vc0));
            have_zt = true;
          }
          float cm = -INFINITY;
          if (nval == 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) cm = fmaxf(cm, __uint_as_float(x[j]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nval) cm = fmaxf(cm, __uint_as_float(x[j]));
          }
          const float mn = fmaxf(m_run, cm);
          const float mL = mn * kLog2e;
          float s0 = 0.0f, s1 = 0.0f;
          if (nval == 32) {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              s0 += ex2_approx(fmaf(__uint_as_float(x[j]), kLog2e, -mL));
              s1 += ex2_approx(fmaf(__uint_as_float(x[j + 1]), kLog2e, -mL));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nval) s0 += ex2_approx(fmaf(__uint_as_float(x[j]), kLog2e, -mL));
          }
          s_run = s_run * ex2_approx((m_run - mn) * kLog2e) + (s0 + s1);
          m_run = mn;
        };
        for (int tt = 0; tt < us.ntiles; ++tt) {
          const uint32_t acc = tile_count & 1u;
          if (!mbar_wait_cl(&tfull[acc], (tile_count >> 1) & 1u, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int64_t vc = us.vb + static_cast<int64_t>(tt) * BN + half * 128;
          const uint32_t ta = lane_base + acc * BN;
          uint32_t xa[32], xb[32];
          tmem_ld_32x32b_x32(ta, xa);
          tmem_ld_wait();
          reg_fence(xa);
          tmem_ld_32x32b_x32(ta + 32, xb);
          chunk(xa, vc);
          tmem_ld_wait();
          reg_fence(xb);
          tmem_ld_32x32b_x32(ta + 64, xa);
          chunk(xb, vc + 32);
          tmem_ld_wait();
          reg_fence(xa);
          tmem_ld_32x32b_x32(ta + 96, xb);
          chunk(xa, vc + 64);
          tmem_ld_wait();
          reg_fence(xb);
          release(acc);
          chunk(xb, vc + 96);
          ++tile_count;
        }
        if (!ok) break;
        // Join the two half-row partials of the warps sharing this lane quarter.
        if (half == 1) {
          if (!mbar_wait(&comb_empty[pq], (items_done & 1u) ^ 1u, wc)) {
            ok = false;
            break;
          }
          comb[pq * 32 + lane] = make_float4(m_run, s_run, zt, have_zt ? 1.0f : 0.0f);
          __syncwarp();
          if (lane == 0) mbar_arrive(&comb_full[pq]);
        } else {
          if (!mbar_wait(&comb_full[pq], items_done & 1u, wc)) {
            ok = false;
            break;
          }
          const float4 o = comb[pq * 32 + lane];
          __syncwarp();
          if (lane == 0) mbar_arrive(&comb_empty[pq]);
          const float M = fmaxf(m_run, o.x);
          float S = 0.0f;
          if (M != -INFINITY)
            S = s_run * ex2_approx((m_run - M) * kLog2e) + o.y * ex2_approx((o.x - M) * kLog2e);
          if (!have_zt && o.w != 0.0f) {
            zt = o.z;
            have_zt = true;
          }
          if (row_ok) {
            a.part[static_cast<int64_t>(t) * a.ug.n_units + u] = make_float2(M, S);
            if (have_zt) a.ztgt[t] = zt;
          }
        }
        ++items_done;
      } else {
        int m_blk, n_blk, row0, col0, part = 0;
        if constexpr (MODE == MODE_GRAD) {
          const MC mc = item_mc(item, a.gm, a.n_mblk, a.n_cols);
          m_blk = mc.m;
          n_blk = mc.c;
          row0 = m_blk * BMP + static_cast<int>(rank) * BM;
          col0 = n_blk * BN + half * 128;   // chunk-local column of this warp's half
        } else {
          n_blk = item % a.n_nblk;
          m_blk = (item / a.n_nblk) % a.n_mblk;
          part = (item / a.n_nblk) / a.n_mblk;   // DH: this item's K part
          row0 = (MODE == MODE_DW ? a.out_row0 : 0) + m_blk * BMP + static_cast<int>(rank) * BM;
          col0 = n_blk * BN + half * 128;
        }
        const int orow = row0 + q * 32;
        const uint32_t acc = tile_count & 1u;
        if (!mbar_wait_cl(&tfull[acc], (tile_count >> 1) & 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        int32_t* flag = nullptr;
        if constexpr (MODE == MODE_DH) {
          // K parts of one tile are added into dH one after the other, in part
          // order, so the sum dH (+)= P0 + P1 + ... is the same at every run.
          // Parts are numbered part-major, so part k - 1 of this tile ran a
          // wave earlier and its count is normally there already.
          if (a.ksplit > 1) {
            flag = a.dh_flags + ((m_blk * a.n_nblk + n_blk) * 2 + static_cast<int>(rank)) * kEpiWarps + e;
            if (part > 0 && !flag_wait_ge(flag, part, lane, wc)) {
              ok = false;
              break;
            }
          }
          add_out = a.accumulate || part > 0;
        }
        const uint32_t ta = lane_base + acc * BN;
        if constexpr (MODE == MODE_GRAD) {
          const int t = m_blk * BMP + static_cast<int>(rank) * BM + r;
          int64_t y = -1;
          float lseL = 0.0f;
          bool row_ok = false;
          if (t < a.pd.T) {
            y = a.targets[t];
            row_ok = (y >= 0) && (y < a.pd.V_real);
            lseL = a.lse[t] * kLog2e;
          }
          const int64_t vt0 = static_cast<int64_t>(a.v0) + col0;
#pragma unroll 1
          for (int bb = 0; bb < 2; ++bb) {
            uint32_t x0[32], x1[32], w[32];
            tmem_ld_32x32b_x32(ta + bb * 64, x0);
            tmem_ld_32x32b_x32(ta + bb * 64 + 32, x1);
            tmem_ld_wait();
            reg_fence(x0);
            reg_fence(x1);
            if (bb == 1) release(acc);
            const int64_t vc0 = vt0 + bb * 64;
            // The chunk's real columns [0, nval) and the target's column jy in
            // it (-1 when elsewhere), fixed for the chunk: the loop below
            // compares only 32-bit column indices. A row without a valid
            // target has no real column and no target column.
            const int64_t nv64 = row_ok ? a.pd.V_real - vc0 : 0;
            const int nval = nv64 >= 64 ? 64 : (nv64 <= 0 ? 0 : static_cast<int>(nv64));
            const int64_t jy64 = y - vc0;
            const int jy = (row_ok && jy64 >= 0 && jy64 < 64) ? static_cast<int>(jy64) : -1;
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              const uint32_t xa = j < 32 ? x0[j] : x1[j - 32];
              const uint32_t xb = j < 32 ? x0[j + 1] : x1[j - 31];
              float g0 = 0.0f, g1 = 0.0f;
              if (j < nval) g0 = ex2_approx(fmaf(__uint_as_float(xa), kLog2e, -lseL)) * scale;
              if (j + 1 < nval) g1 = ex2_approx(fmaf(__uint_as_float(xb), kLog2e, -lseL)) * scale;
              if (j == jy) g0 -= scale;
              if (j + 1 == jy) g1 -= scale;
              w[j / 2] = pack_bf16x2(g0, g1);
            }
            store_box(w, col0 + bb * 64, orow);
          }
        } else {
          uint32_t xa[32], xb[32];
          tmem_ld_32x32b_x32(ta, xa);
          tmem_ld_wait();
          reg_fence(xa);
          tmem_ld_32x32b_x32(ta + 32, xb);
          store_box(xa, col0, orow);
          tmem_ld_wait();
          reg_fence(xb);
          tmem_ld_32x32b_x32(ta + 64, xa);
          store_box(xb, col0 + 32, orow);
          tmem_ld_wait();
          reg_fence(xa);
          tmem_ld_32x32b_x32(ta + 96, xb);
          store_box(xa, col0 + 64, orow);
          tmem_ld_wait();
          reg_fence(xb);
          release(acc);
          store_box(xb, col0 + 96, orow);
          if (MODE == MODE_DH && flag && part + 1 < a.ksplit) {
            // This part's additions are complete in global memory before the
            // next part may add on top of them.
            if (lane == 0) {
              bulk_wait<0>();
              fence_proxy_async_global();
              flag_release(flag, part + 1);
            }
            __syncwarp();
          }
        }
        ++tile_count;
      }
    }
    if constexpr (Tr::staging) {
      if (lane == 0) bulk_wait<0>();
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer's TMEM and shared memory stay live until the pair is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Bounded-wait self-test: one block waits on a barrier nothing completes.
__global__ void wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, status, limit_ns};
    (void)mbar_wait(&bar, 0, wc);
  }
  __syncthreads();
}

// Clusters of this mode that fit on the device at once (asked once per device,
// after the kernel's shared-memory limit has been set there).
template <int MODE>
int max_clusters(const DevInfo& di) {
  static std::atomic<int> cached[64];
  if (di.device < 0 || di.device >= 64) return di.num_sms / 2;
  int n = cached[di.device].load(std::memory_order_acquire);
  if (n > 0) return n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(di.num_sms & ~1), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<MODE>();
  if (cudaOccupancyMaxActiveClusters(&n, tc_loss_kernel<MODE>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return di.num_sms / 2;   // not cached: the query may succeed once the kernel is configured
  }
  cached[di.device].store(n, std::memory_order_release);
  return n;
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& mA, const CUtensorMap& mB, const CUtensorMap& mO, const TcArgs& a,
                        cudaStream_t st) {
  static std::atomic<uint64_t> configured{0};
  if (device_pending(configured)) {
    cudaError_t e = cudaFuncSetAttribute(tc_loss_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes<MODE>()));
    if (e != cudaSuccess) return e;
    mark_device_done(configured);
  }
  if (a.n_items <= 0) return cudaSuccess;
  const DevInfo di = current_device_info();
  const int mc = max_clusters<MODE>(di);
  const int clusters = a.n_items < mc ? a.n_items : mc;
  const cudaError_t e = launch_dependent(tc_loss_kernel<MODE>, dim3(2 * clusters), dim3(kThreads), smem_bytes<MODE>(),
                                         st, mA, mB, mO, a);
  note_launch(MODE == MODE_ARGMAX ? VCE_K_TC_ARGMAX : VCE_K_TC_FWD + MODE, st);
  return e;
}

TcArgs base_args(const vce_problem& p, const int64_t* targets, int32_t* status) {
  TcArgs a{};
  a.pd = prob_dev(p);
  a.targets = targets;
  a.status = status;
  a.limit_ns = wait_limit_ns();
  a.ksplit = 1;
  a.gm = 1;
  a.n_cols = 1;
  return a;
}

// Token blocks per item group (see item_mc): the most whose rows of h fit in
// kGroupBytes, spread evenly over the groups. The Qwen3-like step (32 blocks
// of 1 MB) keeps a single group.
constexpr int64_t kGroupBytes = int64_t(40) << 20;
int tc_group_mblk(const vce_problem& p) {
  const int64_t n_mblk = ceil_div(p.T, BMP);
  if (n_mblk <= 1) return 1;
  int64_t gmax = kGroupBytes / (static_cast<int64_t>(BMP) * p.H * 2);
  if (gmax < 1) gmax = 1;
  const int64_t groups = ceil_div(n_mblk, gmax);
  return static_cast<int>(ceil_div(n_mblk, groups));
}

}  // namespace

// W rows that the units in flight at one time may span: with the token-block
// group's h rows (kGroupBytes) they stay within about half of L2.
constexpr int64_t kUnitWorkingBytes = int64_t(24) << 20;

int tc_unit_width(const vce_problem& p) {
  // The persistent grid takes items in strides of the cluster count; pick the
  // widest unit (fewest partials to merge) whose heaviest cluster carries no
  // more than 1% over the best width's, counting 256-column tiles per item.
  // Widths whose units in flight (about clusters / group size of them) span
  // more than kUnitWorkingBytes of W are passed over while a narrower one
  // stays within it: at H = 3072 a 2048-column unit holds 12.6 MB of W, and
  // the forward ran 3% faster on 1024-column units with the same tile balance.
  const DevInfo di = current_device_info();
  const int64_t clusters = di.num_sms >= 2 ? di.num_sms / 2 : 1;
  const int64_t n_mblk = ceil_div(p.T, BMP);
  if (n_mblk == 0) return kTcUnitWidth;
  struct Memo {
    int64_t T, Vp, V_real, H, clusters;
    int32_t S, uw;
  };
  thread_local Memo memo{-1, -1, -1, -1, -1, -1, 0};
  if (memo.T == p.T && memo.Vp == p.Vp && memo.V_real == p.V_real && memo.H == p.H && memo.S == p.S &&
      memo.clusters == clusters)
    return memo.uw;
  const int gm = tc_group_mblk(p);
  const double units_in_flight = static_cast<double>(clusters) / static_cast<double>(gm < 1 ? 1 : gm);
  int widest = 512;   // the widest width within the working-set bound (512 if none is)
  for (int uw = kTcUnitWidth; uw >= 512; uw -= BN)
    if (units_in_flight * static_cast<double>(uw) * static_cast<double>(p.H) * 2.0 <=
        static_cast<double>(kUnitWorkingBytes)) {
      widest = uw;
      break;
    }
  int best_uw = widest;
  int64_t best_load = -1;
  std::vector<int64_t> load, unit_tiles;
  for (int uw = widest; uw >= 512; uw -= BN) {
    const UnitGrid ug = unit_grid(p, uw);
    unit_tiles.assign(static_cast<size_t>(ug.n_units), 0);
    for (int64_t u = 0; u < ug.n_units; ++u) {
      const int64_t k = u / ug.ups, j = u - k * ug.ups;
      const int64_t lo = shard_lo(k, p.Vp, p.S), hi = shard_lo(k + 1, p.Vp, p.S);
      const int64_t vb = lo + j * uw;
      int64_t ve = vb + uw < hi ? vb + uw : hi;
      if (ve > p.V_real) ve = p.V_real;
      unit_tiles[static_cast<size_t>(u)] = ve > vb ? ceil_div(ve - vb, BN) : 0;
    }
    load.assign(static_cast<size_t>(clusters), 0);
    const int64_t n_items = n_mblk * ug.n_units;
    for (int64_t item = 0; item < n_items; ++item) {   // cluster c takes items c, c + clusters, ...
      const MC mc = item_mc(static_cast<int>(item), gm, static_cast<int>(n_mblk), static_cast<int>(ug.n_units));
      load[static_cast<size_t>(item % clusters)] += unit_tiles[static_cast<size_t>(mc.c)];
    }
    int64_t mx = 0;
    for (int64_t v : load) mx = v > mx ? v : mx;
    if (best_load < 0 || mx * 100 < best_load * 99) {
      best_uw = uw;
      best_load = mx;
    }
  }
  memo = Memo{p.T, p.Vp, p.V_real, p.H, clusters, p.S, best_uw};
  return best_uw;
}

int tc_dh_parts(const vce_problem& p, int vc_act) {
  const DevInfo di = current_device_info();
  const int clusters = max_clusters<MODE_DH>(di);
  const int tiles = static_cast<int>(ceil_div(p.T, BMP) * ceil_div(p.H, BN));
  const int kb = static_cast<int>(ceil_div(vc_act, BK));
  // Fewest parts whose tile count fills the clusters' waves to >= 95%, each
  // part keeping at least 32 K blocks.
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= kMaxDhParts; ++s) {
    if (s > 1 && kb / s < 32) break;
    const int items = tiles * s;
    const int waves = (items + clusters - 1) / clusters;
    const double eff = static_cast<double>(items) / (static_cast<double>(waves) * clusters);
    if (eff > best_eff + 1e-9) {
      best = s;
      best_eff = eff;
    }
    if (eff >= 0.95) break;
  }
  return best;
}

cudaError_t launch_tc_fwd(const vce_problem& p, const UnitGrid& ug, const void* h, const void* W,
                          const int64_t* targets, float2* part, float* ztgt, int32_t* merge_ctr, int32_t* status,
                          cudaStream_t st) {
  CUtensorMap mh, mw;
  if (!make_tmap_2d(&mh, h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, p.T, p.H, 64, BM, true) ||
      !make_tmap_2d(&mw, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, p.V_real, p.H, 64, BNH, true))
    return cudaErrorInvalidValue;
  TcArgs a = base_args(p, targets, status);
  a.n_mblk = static_cast<int>(ceil_div(p.T, BMP));
  a.n_items = a.n_mblk * ug.n_units;
  a.gm = tc_group_mblk(p);
  a.n_cols = ug.n_units;
  a.num_kb = static_cast<int>(ceil_div(p.H, BK));
  a.ug = ug;
  a.part = part;
  a.ztgt = ztgt;
  a.merge_ctr = merge_ctr;
  return launch_mode<MODE_FWD>(mh, mw, mh, a, st);
}

cudaError_t launch_tc_argmax(const vce_problem& p, const UnitGrid& ug, const void* h, const void* W, float2* part,
                             int32_t* status, cudaStream_t st) {
  CUtensorMap mh, mw;
  if (!make_tmap_2d(&mh, h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, p.T, p.H, 64, BM, true) ||
      !make_tmap_2d(&mw, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.H, p.V_real, p.H, 64, BNH, true))
    return cudaErrorInvalidValue;
  TcArgs a = base_args(p, nullptr, status);
  a.n_mblk = static_cast<int>(ceil_div(p.T, BMP));
  a.n_items = a.n_mblk * ug.n_units;
  a.gm = tc_group_mblk(p);
  a.n_cols = ug.n_units;
  a.num_kb = static_cast<int>(ceil_div(p.H, BK));
  a.ug = ug;
  a.part = part;
  return launch_mode<MODE_ARGMAX>(mh, mw, mh, a, st);
}

cudaError_t launch_tc_bwd_chunk(const vce_problem& p, const void* h, const void* W, const int64_t* targets,
                                const float* lse, float g, int v0, int vc_act, void* G,
                                int g_ld, float* dH, bool dH_accumulate, float* dW, bool dW_accumulate,
                                int32_t* dh_flags, int dh_parts, int32_t* status, cudaStream_t st) {
  const int parts = dh_flags ? dh_parts : 1;
  const int n_flags = static_cast<int>(ceil_div(p.T, BMP) * ceil_div(p.H, BN)) * 2 * kEpiWarps;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cudaError_t e;
  // GRAD: G[:, 0:vc_act] for vocabulary columns [v0, v0 + vc_act).
  {
    CUtensorMap mh, mw, mg;
    if (!make_tmap_2d(&mh, h, BF, 2, p.H, p.T, p.H, 64, BM, true) ||
        !make_tmap_2d(&mw, W, BF, 2, p.H, p.V_real, p.H, 64, BNH, true) ||
        !make_tmap_2d(&mg, G, BF, 2, vc_act, p.T, g_ld, 64, 32, true))
      return cudaErrorInvalidValue;
    TcArgs a = base_args(p, targets, status);
    a.n_mblk = static_cast<int>(ceil_div(p.T, BMP));
    a.n_nblk = static_cast<int>(ceil_div(vc_act, BN));
    a.n_items = a.n_mblk * a.n_nblk;
    a.gm = tc_group_mblk(p);
    a.n_cols = a.n_nblk;
    a.num_kb = static_cast<int>(ceil_div(p.H, BK));
    a.lse = lse;
    a.g = g;
    a.v0 = v0;
    a.vc = vc_act;
    a.dh_flags = parts > 1 ? dh_flags : nullptr;
    a.n_dh_flags = parts > 1 ? n_flags : 0;
    if ((e = launch_mode<MODE_GRAD>(mh, mw, mg, a, st)) != cudaSuccess) return e;
  }
  // DH: dH (+)= G[:, 0:vc_act] W[v0:v0+vc_act, :]. With dh_parts > 1 the K
  // range is cut into parts; each part's tile is added into dH after the part
  // before it (counters in dh_flags), so the order of the additions is fixed.
  {
    CUtensorMap mg, mw, mo;
    if (!make_tmap_2d(&mg, G, BF, 2, vc_act, p.T, g_ld, 64, BM, true) ||
        !make_tmap_2d(&mw, W, BF, 2, p.H, p.V_real, p.H, 64, 64, true) ||
        !make_tmap_2d(&mo, dH, F32, 4, p.H, p.T, p.H, 32, 32, true))
      return cudaErrorInvalidValue;
    TcArgs a = base_args(p, targets, status);
    a.n_mblk = static_cast<int>(ceil_div(p.T, BMP));
    a.n_nblk = static_cast<int>(ceil_div(p.H, BN));
    a.num_kb = static_cast<int>(ceil_div(vc_act, BK));
    a.ksplit = parts;
    a.kb_per = static_cast<int>(ceil_div(a.num_kb, parts));
    a.dh_flags = parts > 1 ? dh_flags : nullptr;
    a.n_dh_flags = parts > 1 ? n_flags : 0;
    a.n_items = a.n_mblk * parts * a.n_nblk;
    a.v0 = v0;
    a.accumulate = dH_accumulate ? 1 : 0;
    if ((e = launch_mode<MODE_DH>(mg, mw, mo, a, st)) != cudaSuccess) return e;
  }
  // DW: dW[v0:v0+vc_act, :] (+)= G[:, 0:vc_act]^T h
  {
    CUtensorMap mg, mh, mo;
    if (!make_tmap_2d(&mg, G, BF, 2, vc_act, p.T, g_ld, 64, 64, true) ||
        !make_tmap_2d(&mh, h, BF, 2, p.H, p.T, p.H, 64, 64, true) ||
        !make_tmap_2d(&mo, dW, F32, 4, p.H, static_cast<uint64_t>(v0) + vc_act, p.H, 32, 32, true))
      return cudaErrorInvalidValue;
    TcArgs a = base_args(p, targets, status);
    a.n_mblk = static_cast<int>(ceil_div(vc_act, BMP));
    a.n_nblk = static_cast<int>(ceil_div(p.H, BN));
    a.n_items = a.n_mblk * a.n_nblk;
    a.num_kb = static_cast<int>(ceil_div(p.T, BK));
    a.out_row0 = v0;
    a.accumulate = dW_accumulate ? 1 : 0;
    if ((e = launch_mode<MODE_DW>(mg, mh, mo, a, st)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, int32_t* status, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  note_launch(VCE_K_WAIT_SELFTEST, st);
  return cudaGetLastError();
}

}  // namespace vce
