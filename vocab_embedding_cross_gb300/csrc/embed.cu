// Vocabulary-sharded embedding: masked lookup and deterministic backward.
//
// Forward ("Vocabulary shards: look up locally and normalize globally",
// paragraph 1; "Tensor Parallelism (TP)", Embedding): the ownership test is
// made on the global id before any row address is formed. A valid id is owned
// by exactly one shard, so the sum of the S masked partial lookups is the
// owner's row; on one GPU that sum is the row itself, copied with 16-byte
// vector loads. Invalid ids (padding id, negatives, padded rows, >= Vp) give
// zero rows.
//
// Backward (same page, paragraph 2: repeated tokens accumulate into the same
// owned row): the valid (id, t) pairs are sorted stably by id (for T <= 16384
// one CTA per SM sorts the ids with id mod NB equal to its index, its CTAs
// grouped in clusters that share the id loads above 8192 tokens; otherwise one
// CTA sorts 64-bit keys), the tokens of each id are cut into runs of
// kEmbedBwdChunk, each run is summed in fp32 in ascending t, run sums are
// combined left to right, and the total is added once into the fp32 row. The
// order is fixed, so results are bit-identical from run to run.
//
// The sort depends on the ids alone. It leaves a plan in the workspace (the
// sorted tokens, the run descriptors, zeroed combine counters and a header
// that names the problem's shape), and the reduce applies the plan to dE. The
// reduce leaves the plan as it found it, so one plan can be applied again, and
// a plan can be made as soon as the ids are known, before dE exists.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <type_traits>

#include "internal.h"

namespace vce {
namespace {


// ---------------------------------------------------------------------------
// Forward gather: one warp per token row.
// ---------------------------------------------------------------------------
constexpr int kGatherWarps = 8;

// BESIDE_PLAN: launched as a dependent of the backward's plan (the sort), which
// it does not read, so that it runs beside the sort on the SMs the sort leaves
// free. Its last CTA waits for the sort to end before exiting, so the lookup
// completes only after the plan does and a kernel that waits for the lookup
// also sees the plan.
template <bool BESIDE_PLAN>
__global__ void __launch_bounds__(kGatherWarps * 32)
    embed_gather_kernel(const int64_t* __restrict__ ids, const uint4* __restrict__ W, uint4* __restrict__ E,
                        int32_t* __restrict__ owner, int32_t* __restrict__ local, int64_t T, int64_t Vp,
                        int64_t V_real, int32_t S, int row_vecs) {
  if constexpr (BESIDE_PLAN) {
    if (blockIdx.x == gridDim.x - 1) grid_dep_wait();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kGatherWarps + warp;
  if (t >= T) return;
  const int64_t id = __ldg(ids + t);
  const bool valid = (id >= 0) && (id < V_real);   // ownership test before indexing
  if (lane == 0) {
    int32_t k = -1, l = -1;
    if (valid) {
      k = shard_of(id, Vp, S);
      l = static_cast<int32_t>(id - shard_lo(k, Vp, S));
    }
    if (owner) owner[t] = k;
    if (local) local[t] = l;
  }
  uint4* dst = E + t * row_vecs;
  if (!valid) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int i = lane; i < row_vecs; i += 32) dst[i] = z;
    return;
  }
  const uint4* src = W + id * row_vecs;
  int i = lane;
  for (; i + 96 < row_vecs; i += 128) {
    uint4 a = __ldg(src + i), b = __ldg(src + i + 32), c = __ldg(src + i + 64), d = __ldg(src + i + 96);
    dst[i] = a;
    dst[i + 32] = b;
    dst[i + 64] = c;
    dst[i + 96] = d;
  }
  for (; i < row_vecs; i += 32) dst[i] = __ldg(src + i);
}

// ---------------------------------------------------------------------------
// Backward, step 1: one CTA sorts the valid (id, t) keys and builds the runs.
// Two variants: keys in shared memory (T <= 16384 and id, t packed in 32 bits)
// and keys in the workspace (any size, 64-bit keys). Both leave the sorted
// token indices in `tsorted` and the run descriptors in `runs`.
// ---------------------------------------------------------------------------
constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 8;
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kRadix = 256;
constexpr int kSmemSortMax = 16384;                       // keys the shared-memory variant holds
constexpr int kSmemItems = kSmemSortMax / kSortThreads;   // at most 16 rounds of 32 keys per warp
constexpr int kSortDigitBits = 9;                         // radix of the shared-memory passes
constexpr int kSortDigits = 1 << kSortDigitBits;
// Shared-memory arrays are padded by one word per 32 (index i at i + i/32), so
// that each thread's 16 consecutive entries fall in distinct banks across a warp.
__host__ __device__ constexpr int pad32(int i) { return i + (i >> 5); }
constexpr size_t kSmemSortBytes = 2 * pad32(kSmemSortMax) * sizeof(uint32_t) +
                                  kSortWarps * kSortDigits * sizeof(int) + 64 * sizeof(int);

struct __align__(16) RunDesc {
  int32_t start, end;   // sorted positions [start, end)
  int32_t id;
  int32_t slot;         // partial slot (multi-run ids) or -1
  int32_t mseg;         // index of the multi-run id, or -1
  int32_t nruns;        // runs of this id
  int32_t first_slot;   // slot of the id's first run
  int32_t pad;
};

// The workspace header (16 words). The sorts claim space with atomic
// additions on words 0-5; the reduce hands out items from word 6; words 8-11
// describe the plan (its T, the column slices per row of its multi-run ids'
// counters, a marker and the number of rows its ids index), so that applying
// a plan made for another shape or slice width, or a workspace that holds
// none, is refused on the device before any row is touched.
constexpr int kHdrItem = 6, kHdrPlanT = 8, kHdrPlanNh = 9, kHdrPlanMark = 10, kHdrPlanRows = 11;
constexpr int32_t kPlanMark = 0x4E414C50;   // "PLAN"

__device__ __forceinline__ void plan_seal(int32_t* hdr, int T, int nhm, int64_t V_real) {
  hdr[kHdrPlanT] = T;
  hdr[kHdrPlanNh] = nhm;
  hdr[kHdrPlanRows] = static_cast<int32_t>(V_real);
  hdr[kHdrPlanMark] = kPlanMark;
}

struct BwdLayout {
  size_t hdr, keys_a, keys_b, seg_start, tsorted, runs, counters, partials, total;
  int64_t n_counters, n_slots;
  int nh;    // wide column slices per row: the items of single-run ids
  int nhm;   // narrow column slices (half as wide): the items and counters of multi-run ids
};

int cols_per_item(int esize) { return 128 * (16 / esize); }

BwdLayout bwd_layout(const vce_problem& p) {
  BwdLayout L{};
  const int64_t T = p.T;
  const int esize = p.dtype == VCE_BF16 ? 2 : 4;
  L.nh = static_cast<int>(ceil_div(p.H, cols_per_item(esize)));
  L.nhm = static_cast<int>(ceil_div(p.H, cols_per_item(esize) / 2));
  L.n_counters = (T / (kEmbedBwdChunk + 1) + 2) * L.nhm;
  L.n_slots = 2 * T / kEmbedBwdChunk + 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, kWsAlign);
    return o;
  };
  L.hdr = take(64);
  L.keys_a = take(sizeof(uint64_t) * (T + 1));
  L.keys_b = take(sizeof(uint64_t) * (T + 1));
  L.seg_start = take(sizeof(int32_t) * (T + 2));
  L.tsorted = take(sizeof(int32_t) * (T + 1));
  L.runs = take(sizeof(RunDesc) * (T + 1));
  L.counters = take(sizeof(int32_t) * L.n_counters);
  L.partials = take(sizeof(float) * L.n_slots * p.H);
  L.total = off;
  return L;
}

int bit_width(int64_t x) {   // bits needed for values in [0, x)
  int b = 1;
  while (b < 62 && (int64_t(1) << b) < x) ++b;
  return b;
}

// Block-wide exclusive scan of one int per thread (up to 1024 threads).
__device__ __forceinline__ int block_excl_scan(int v, int* sh_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < static_cast<int>(blockDim.x >> 5) ? sh_warp[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh_warp[lane] = s - w;          // exclusive prefix of warp totals
    if (lane == 31) sh_warp[32] = s;
  }
  __syncthreads();
  const int res = sh_warp[warp] + x - v;
  *total = sh_warp[32];
  __syncthreads();
  return res;
}

// The same scan over 64-bit values (four 16-bit counters packed in one word).
__device__ __forceinline__ uint64_t block_excl_scan64(uint64_t v, uint64_t* sh_warp, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint64_t w = lane < static_cast<int>(blockDim.x >> 5) ? sh_warp[lane] : 0;
    uint64_t s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh_warp[lane] = s - w;
    if (lane == 31) sh_warp[32] = s;
  }
  __syncthreads();
  const uint64_t res = sh_warp[warp] + x - v;
  *total = sh_warp[32];
  __syncthreads();
  return res;
}

// Runs of kEmbedBwdChunk tokens for the segments [s0, s0 + per_thread) of one
// thread (all threads together cover [0, nseg) in order); slots for multi-run
// ids. seg[s] is the sorted position where segment s starts (segment s ends at
// seg[s + 1], the last one at n); id_of(s) gives its id. As in the bucketed
// sorts, the runs of multi-run ids go to the front of the run list (at their
// slot's index) and single runs to its back (from index cap - 1 down).
template <typename SegAt, typename IdOf>
__device__ __forceinline__ void build_runs(SegAt seg, int nseg, int n, int cap, int per_thread, int nhm, IdOf id_of,
                                           int* sh_warp, int32_t* hdr, RunDesc* runs, int32_t* counters) {
  const int s0 = threadIdx.x * per_thread;
  int my_runs = 0, my_multi = 0, my_slots = 0;
  for (int j = 0; j < per_thread; ++j) {
    const int s = s0 + j;
    if (s < nseg) {
      const int en = s + 1 < nseg ? seg(s + 1) : n;
      const int nr = (en - seg(s) + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
      my_runs += nr;
      if (nr > 1) {
        my_multi += 1;
        my_slots += nr;
      }
    }
  }
  int t_runs, t_multi, t_slots;
  block_excl_scan(my_runs, sh_warp, &t_runs);
  int m0 = block_excl_scan(my_multi, sh_warp, &t_multi);
  int q0 = block_excl_scan(my_slots, sh_warp, &t_slots);
  int sb = min(s0, nseg) - m0;   // single-run segments before this thread's
  for (int j = 0; j < per_thread; ++j) {
    const int s = s0 + j;
    if (s >= nseg) break;
    const int st = seg(s), en = s + 1 < nseg ? seg(s + 1) : n;
    const int nr = (en - st + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    const bool multi = nr > 1;
    const int id = id_of(s);
    for (int k = 0; k < nr; ++k) {
      RunDesc r;
      r.start = st + k * kEmbedBwdChunk;
      r.end = min(en, st + (k + 1) * kEmbedBwdChunk);
      r.id = id;
      r.slot = multi ? q0 + k : -1;
      r.mseg = multi ? m0 : -1;
      r.nruns = nr;
      r.first_slot = multi ? q0 : -1;
      r.pad = 0;
      // multi-run ids' runs at the front (index = slot), single runs at the back
      runs[multi ? q0 + k : cap - 1 - sb] = r;
    }
    if (multi) {
      for (int hh = 0; hh < nhm; ++hh) counters[m0 * nhm + hh] = 0;
      m0 += 1;
      q0 += nr;
    } else {
      sb += 1;
    }
  }
  if (threadIdx.x == 0) {
    hdr[1] = t_slots;   // runs at the front
    hdr[3] = t_multi;
    hdr[4] = t_slots;
    hdr[5] = nseg - t_multi;   // single runs at the back
    hdr[kHdrItem] = 0;   // the reduce's item counter
  }
}

// Shared-memory variant: keys (id << tbits) | t in 32 bits, T <= kSmemSortMax.
__global__ void __launch_bounds__(kSortThreads, 1)
    embed_sort_smem_kernel(const int64_t* __restrict__ ids, int T, int64_t V_real, int tbits, int idbits, int nhm,
                           int32_t* hdr, int32_t* tsorted, RunDesc* runs, int32_t* counters) {
  extern __shared__ __align__(16) uint32_t smem_keys[];
  uint32_t* ka = smem_keys;
  uint32_t* kb = smem_keys + pad32(kSmemSortMax);
  int* ctab = reinterpret_cast<int*>(smem_keys + 2 * pad32(kSmemSortMax));   // [32 warps][512 digits]
  int* sh_warp = ctab + kSortWarps * kSortDigits;                              // 64 ints
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;

  // Phase 0: stable compaction of the valid ids. Warp w reads its contiguous
  // block of tokens 32 at a time (coalesced, all loads issued before use);
  // ballots give the order.
  const int tpw = ((T + kSortWarps - 1) / kSortWarps + 31) / 32 * 32;   // tokens per warp, <= 512
  constexpr uint32_t kNoKey = 0xFFFFFFFFu;
  uint32_t tkey[kSmemItems];
#pragma unroll
  for (int j = 0; j < kSmemItems; ++j) {
    const int t = warp * tpw + j * 32 + lane;
    const int64_t id = (j < tpw / 32 && t < T) ? ids[t] : -1;
    tkey[j] = (id >= 0 && id < V_real) ? (static_cast<uint32_t>(id) << tbits) | static_cast<uint32_t>(t) : kNoKey;
  }
  int wcount = 0;
#pragma unroll
  for (int j = 0; j < kSmemItems; ++j) wcount += __popc(__ballot_sync(0xffffffffu, tkey[j] != kNoKey));
  if (lane == 0) sh_warp[warp] = wcount;
  __syncthreads();
  int wbase = 0, n = 0;
  for (int w = 0; w < kSortWarps; ++w) {
    const int c = sh_warp[w];
    wbase += w < warp ? c : 0;
    n += c;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kSmemItems; ++j) {
    const bool ok = tkey[j] != kNoKey;
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (ok) ka[pad32(wbase + __popc(bal & lt_mask))] = tkey[j];
    wbase += __popc(bal);
  }
  __syncthreads();

  // Phase 1: stable LSD radix passes over the id bits, 9 bits per pass. Warp
  // w owns the kpw consecutive keys [w*kpw, (w+1)*kpw) and takes them 32 at a
  // time; lanes holding the same digit find each other with one ballot per
  // digit bit, which gives each key its rank among the warp's keys of that
  // digit (in key order). The per-warp digit counts are then scanned digit-major, warp-minor,
  // so every key lands at a stable position.
  const int kpw = ((n + kSortWarps - 1) / kSortWarps + 31) & ~31;   // keys per warp, <= 512
  const int rounds = kpw >> 5;                                      // <= 16
  int* whist = ctab + warp * kSortDigits;                            // this warp's digit counts
  uint32_t* src = ka;
  uint32_t* dst = kb;
  for (int shift = tbits; shift < tbits + idbits; shift += kSortDigitBits) {
    for (int i = tid; i < kSortWarps * kSortDigits; i += kSortThreads) ctab[i] = 0;
    __syncthreads();
    uint32_t key[kSmemItems];
    uint32_t rk[kSmemItems / 2] = {};   // 16-bit ranks, two per word
#pragma unroll
    for (int j = 0; j < kSmemItems; ++j) {
      if (j < rounds) {
        const int q = warp * kpw + j * 32 + lane;
        const bool ok = q < n;
        key[j] = ok ? src[pad32(q)] : 0u;
        const uint32_t d = ok ? (key[j] >> shift) & (kSortDigits - 1) : kSortDigits;
        uint32_t peers = __ballot_sync(0xffffffffu, ok);
#pragma unroll
        for (int b = 0; b < kSortDigitBits; ++b) {
          const uint32_t bb = __ballot_sync(0xffffffffu, (d >> b) & 1u);
          peers &= ((d >> b) & 1u) ? bb : ~bb;
        }
        int base = 0;
        if (ok) base = whist[d];
        __syncwarp();
        if (ok) {
          rk[j >> 1] |= static_cast<uint32_t>(base + __popc(peers & lt_mask)) << ((j & 1) * 16);
          if (lane == __ffs(peers) - 1) whist[d] = base + __popc(peers);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    {
      // Thread tid scans digit tid/2 over warps [16*(tid&1), +16).
      const int d = tid >> 1, w0 = (tid & 1) * 16;
      int v[16];
      int sum = 0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        v[k] = ctab[(w0 + k) * kSortDigits + d];
        sum += v[k];
      }
      int all;
      int run = block_excl_scan(sum, sh_warp, &all);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        ctab[(w0 + k) * kSortDigits + d] = run;
        run += v[k];
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kSmemItems; ++j) {
      const int q = warp * kpw + j * 32 + lane;
      if (j < rounds && q < n) {
        const int d = static_cast<int>((key[j] >> shift) & (kSortDigits - 1));
        dst[pad32(whist[d] + static_cast<int>((rk[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu))] = key[j];
      }
    }
    __syncthreads();
    uint32_t* tmp = src;
    src = dst;
    dst = tmp;
  }

  // Phase 2: sorted token indices to global memory (coalesced within each
  // warp's chunk) and the segment heads (first position of every distinct id)
  // into the free key buffer.
  const uint32_t tmask = (1u << tbits) - 1u;
  int* seg = reinterpret_cast<int*>(dst);
  auto is_head = [&](int q) { return q == 0 || (src[pad32(q)] >> tbits) != (src[pad32(q - 1)] >> tbits); };
  int wheads = 0;
  for (int j = 0; j < rounds; ++j) {
    const int q = warp * kpw + j * 32 + lane;
    const bool ok = q < n;
    if (ok) tsorted[q] = static_cast<int32_t>(src[pad32(q)] & tmask);
    wheads += __popc(__ballot_sync(0xffffffffu, ok && is_head(q)));
  }
  if (lane == 0) sh_warp[32 + warp] = wheads;
  __syncthreads();
  int hbase = 0, nseg = 0;
  for (int w = 0; w < kSortWarps; ++w) {
    const int c = sh_warp[32 + w];
    hbase += w < warp ? c : 0;
    nseg += c;
  }
  for (int j = 0; j < rounds; ++j) {
    const int q = warp * kpw + j * 32 + lane;
    const bool h = q < n && is_head(q);
    const uint32_t bal = __ballot_sync(0xffffffffu, h);
    if (h) seg[pad32(hbase + __popc(bal & lt_mask))] = q;
    hbase += __popc(bal);
  }
  __syncthreads();

  // Phase 3: runs of kEmbedBwdChunk tokens. Warp w takes segments
  // [w*spw, (w+1)*spw), one per lane per round; a block scan of the warps'
  // (runs, multi-run segments) totals gives each segment its first run and
  // first partial slot, and the lane holding a segment writes its runs: a
  // multi-run id's at the front of the list, a single run at its back.
  auto seg_end = [&](int sg) { return sg + 1 < nseg ? seg[pad32(sg + 1)] : n; };
  const int spw = ((nseg + kSortWarps - 1) / kSortWarps + 31) & ~31;
  int wpacked = 0;   // (runs << 16) | multi-run segments, over this warp's segments
  for (int j = 0; j < spw; j += 32) {
    const int sg = warp * spw + j + lane;
    int pk = 0;
    if (sg < nseg) {
      const int nr = (seg_end(sg) - seg[pad32(sg)] + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
      pk = (nr << 16) | (nr > 1 ? 1 : 0);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pk += __shfl_xor_sync(0xffffffffu, pk, o);
    wpacked += pk;
  }
  int tot_packed;
  int pre = block_excl_scan(lane == 0 ? wpacked : 0, sh_warp, &tot_packed);
  pre = __shfl_sync(0xffffffffu, pre, 0);
  const int n_runs = tot_packed >> 16, n_multi = tot_packed & 0xFFFF;
  for (int j = 0; j < spw; j += 32) {
    const int sg = warp * spw + j + lane;
    int nr = 0, st = 0, en = 0;
    if (sg < nseg) {
      st = seg[pad32(sg)];
      en = seg_end(sg);
      nr = (en - st + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    }
    const int pk = sg < nseg ? (nr << 16) | (nr > 1 ? 1 : 0) : 0;
    int incl = pk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int mine = pre + incl - pk;   // packed prefix before this segment
    pre += __shfl_sync(0xffffffffu, incl, 31);
    if (sg < nseg) {
      const int rb = mine >> 16, mb = mine & 0xFFFF;
      const bool multi = nr > 1;
      const int q0 = rb - (sg - mb);   // slots used by the multi-run segments before sg
      const int32_t id = static_cast<int32_t>(src[pad32(st)] >> tbits);
      for (int k = 0; k < nr; ++k) {
        RunDesc rd;
        rd.start = st + k * kEmbedBwdChunk;
        rd.end = min(en, rd.start + kEmbedBwdChunk);
        rd.id = id;
        rd.slot = multi ? q0 + k : -1;
        rd.mseg = multi ? mb : -1;
        rd.nruns = nr;
        rd.first_slot = multi ? q0 : -1;
        rd.pad = 0;
        // multi-run ids' runs at the front (index = slot), single runs at the
        // back (sg - mb single segments before this one)
        runs[multi ? q0 + k : T - 1 - (sg - mb)] = rd;
      }
      if (multi)
        for (int hh = 0; hh < nhm; ++hh) counters[mb * nhm + hh] = 0;
    }
  }
  if (tid == 0) {
    hdr[0] = n;
    hdr[1] = n_runs - (nseg - n_multi);   // runs at the front: the slots
    hdr[2] = nseg;
    hdr[3] = n_multi;
    hdr[4] = n_runs - (nseg - n_multi);
    hdr[5] = nseg - n_multi;              // single runs at the back
    hdr[kHdrItem] = 0;   // the reduce's item counter
    plan_seal(hdr, T, nhm, V_real);
  }
}

// Zeroes the workspace headers (up to three; null ones are skipped) that the
// bucketed sorts' CTAs claim space from. It lets its dependent (the first sort)
// start at once: a sort loads and filters its ids, then waits for the kernel
// before it before its first claim.
__global__ void embed_hdr_zero_kernel(int32_t* h0, int32_t* h1, int32_t* h2) {
  grid_dep_launch();
  const int i = threadIdx.x & 15, k = threadIdx.x >> 4;
  int32_t* h = k == 0 ? h0 : (k == 1 ? h1 : h2);
  if (k < 3 && h) h[i] = 0;
}


// Bucketed variant: the sort spread over gridDim.x CTAs (one per SM). CTA b
// takes the valid ids with id % NB == b, in token order, and sorts them by
// id / NB (stable LSD radix, 6-bit digits, warp-level ranking by ballots) in
// shared memory. It then cuts its ids into runs exactly as the single-CTA
// variants do and claims space for its sorted tokens, runs and partial slots
// with atomic additions on the header, which a kernel zeroes first. The
// order of the buckets in the arrays depends on which CTA claims first; every
// id's runs and their order do not, so the reduce gives the same bits.
constexpr int kBktThreads = 1024;
constexpr int kBktWarps = kBktThreads / 32;
constexpr int kBktDigitBits = 6;
constexpr int kBktDigits = 1 << kBktDigitBits;

size_t bucket_sort_smem(int64_t T) {   // two key buffers, 16-bit ranks (whole words), digit counts, scratch
  return static_cast<size_t>(T) * 2 * sizeof(uint32_t) + static_cast<size_t>((T + 1) / 2) * sizeof(uint32_t) +
         kBktWarps * kBktDigits * sizeof(int) + 96 * sizeof(int);
}

__global__ void __launch_bounds__(kBktThreads, 1)
    embed_sort_bucket_kernel(const int64_t* __restrict__ ids, int T, int64_t V_real, int tbits, int qbits, int nhm,
                             uint32_t nb_magic, int32_t* hdr, int32_t* tsorted, RunDesc* runs,
                             int32_t* counters) {
  extern __shared__ __align__(16) uint32_t bsm[];
  uint32_t* ka = bsm;
  uint32_t* kb = bsm + T;
  uint16_t* rank16 = reinterpret_cast<uint16_t*>(bsm + 2 * T);
  int* hist = reinterpret_cast<int*>(bsm + 2 * T + (T + 1) / 2);   // [warps][64 digits]
  // 96 ints of scratch: [0, 32) per-warp counts, [32, 65) the block scan, [80, 84) broadcasts
  int* sh = hist + kBktWarps * kBktDigits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const uint32_t NB = gridDim.x, b = blockIdx.x;

  grid_dep_launch();   // the reduce may be scheduled from here on; it waits for this grid to end

  // Phase A: this bucket's ids in token order. Warp w scans tokens
  // [w*tpw, (w+1)*tpw) 32 at a time; ballots give the order. Every id a
  // thread needs is loaded before any is used, so the loads are in flight
  // together.
  const int tpw = ((T + kBktWarps - 1) / kBktWarps + 31) & ~31;
  constexpr int kMaxRounds = kSmemSortMax / kBktWarps / 32;   // 16 rounds of 32 tokens per warp at most
  int64_t idv[kMaxRounds];
#pragma unroll
  for (int j = 0; j < kMaxRounds; ++j) {
    const int t = warp * tpw + j * 32 + lane;
    idv[j] = (j * 32 < tpw && t < T) ? __ldg(ids + t) : -1;
  }
  uint32_t tkey[kMaxRounds];
#pragma unroll
  for (int j = 0; j < kMaxRounds; ++j) {
    uint32_t k = 0xFFFFFFFFu;
    if (idv[j] >= 0 && idv[j] < V_real) {
      const uint32_t u = static_cast<uint32_t>(idv[j]);
      const uint32_t q = __umulhi(u, nb_magic);   // u / NB, exact for u < 2^32 / NB
      if (u - q * NB == b) k = (q << tbits) | static_cast<uint32_t>(warp * tpw + j * 32 + lane);
    }
    tkey[j] = k;
  }
  int wcount = 0;
#pragma unroll
  for (int j = 0; j < kMaxRounds; ++j) wcount += __popc(__ballot_sync(0xffffffffu, tkey[j] != 0xFFFFFFFFu));
  if (lane == 0) sh[warp] = wcount;
  __syncthreads();
  int wbase = 0, m = 0;
  for (int w = 0; w < kBktWarps; ++w) {
    const int c = sh[w];
    wbase += w < warp ? c : 0;
    m += c;
  }
#pragma unroll
  for (int j = 0; j < kMaxRounds; ++j) {
    const bool ok = tkey[j] != 0xFFFFFFFFu;
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (ok) ka[wbase + __popc(bal & lt_mask)] = tkey[j];
    wbase += __popc(bal);
  }
  // This bucket's place in tsorted. The header is zeroed by the kernel before
  // this one; the claim's result is first needed after phase B, so its round
  // trip overlaps the passes.
  grid_dep_wait();
  int tb = 0;
  if (tid == 0 && m > 0) tb = atomicAdd(&hdr[0], m);
  if (tid == 0 && b == 0) plan_seal(hdr, T, nhm, V_real);

  // Phase B: stable LSD radix passes over the id / NB bits.
  const int kpw = ((m + kBktWarps - 1) / kBktWarps + 31) & ~31;
  int* whist = hist + warp * kBktDigits;
  uint32_t* src = ka;
  uint32_t* dst = kb;
  for (int shift = tbits; shift < tbits + qbits; shift += kBktDigitBits) {
    for (int i = tid; i < kBktWarps * kBktDigits; i += kBktThreads) hist[i] = 0;
    __syncthreads();
    for (int j = 0; j < kpw; j += 32) {
      const int q = warp * kpw + j + lane;
      const bool ok = q < m;
      const uint32_t d = ok ? (src[q] >> shift) & (kBktDigits - 1) : kBktDigits;
      uint32_t peers = __ballot_sync(0xffffffffu, ok);
#pragma unroll
      for (int bit = 0; bit < kBktDigitBits; ++bit) {
        const uint32_t bb = __ballot_sync(0xffffffffu, (d >> bit) & 1u);
        peers &= ((d >> bit) & 1u) ? bb : ~bb;
      }
      int base = 0;
      if (ok) base = whist[d];
      __syncwarp();
      if (ok) {
        rank16[q] = static_cast<uint16_t>(base + __popc(peers & lt_mask));
        if (lane == __ffs(peers) - 1) whist[d] = base + __popc(peers);
      }
      __syncwarp();
    }
    __syncthreads();
    {
      // digits x warps, digit-major, two entries per thread: thread tid takes
      // digit tid / (warps/2) and warps 2 * (tid % (warps/2)), +1.
      static_assert(kBktWarps * kBktDigits == 2 * kBktThreads, "two scan entries per thread");
      const int d = tid / (kBktWarps / 2), w0 = (tid % (kBktWarps / 2)) * 2;
      const int v0 = hist[w0 * kBktDigits + d], v1 = hist[(w0 + 1) * kBktDigits + d];
      int all;
      const int run = block_excl_scan(v0 + v1, sh + 32, &all);
      hist[w0 * kBktDigits + d] = run;
      hist[(w0 + 1) * kBktDigits + d] = run + v0;
    }
    __syncthreads();
    for (int j = 0; j < kpw; j += 32) {
      const int q = warp * kpw + j + lane;
      if (q < m) {
        const uint32_t k = src[q];
        dst[whist[(k >> shift) & (kBktDigits - 1)] + rank16[q]] = k;
      }
    }
    __syncthreads();
    uint32_t* tmp = src;
    src = dst;
    dst = tmp;
  }

  if (tid == 0) sh[80] = tb;
  __syncthreads();
  const int tbase = sh[80];

  // Phase C: sorted tokens, segment heads, runs.
  const uint32_t tmask = (1u << tbits) - 1u;
  int* seg = reinterpret_cast<int*>(dst);
  auto is_head = [&](int q) { return q == 0 || (src[q] >> tbits) != (src[q - 1] >> tbits); };
  int wheads = 0;
  for (int j = 0; j < kpw; j += 32) {
    const int q = warp * kpw + j + lane;
    const bool ok = q < m;
    if (ok) tsorted[tbase + q] = static_cast<int32_t>(src[q] & tmask);
    wheads += __popc(__ballot_sync(0xffffffffu, ok && is_head(q)));
  }
  if (lane == 0) sh[warp] = wheads;
  __syncthreads();
  int hbase = 0, nseg = 0;
  for (int w = 0; w < kBktWarps; ++w) {
    const int c = sh[w];
    hbase += w < warp ? c : 0;
    nseg += c;
  }
  for (int j = 0; j < kpw; j += 32) {
    const int q = warp * kpw + j + lane;
    const bool h = q < m && is_head(q);
    const uint32_t bal = __ballot_sync(0xffffffffu, h);
    if (h) seg[hbase + __popc(bal & lt_mask)] = q;
    hbase += __popc(bal);
  }
  __syncthreads();
  auto seg_end = [&](int sg) { return sg + 1 < nseg ? seg[sg + 1] : m; };
  const int spw = ((nseg + kBktWarps - 1) / kBktWarps + 31) & ~31;
  int wpacked = 0;   // (runs << 16) | multi-run segments, over this warp's segments
  for (int j = 0; j < spw; j += 32) {
    const int sg = warp * spw + j + lane;
    int pk = 0;
    if (sg < nseg) {
      const int nr = (seg_end(sg) - seg[sg] + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
      pk = (nr << 16) | (nr > 1 ? 1 : 0);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pk += __shfl_xor_sync(0xffffffffu, pk, o);
    wpacked += pk;
  }
  int tot_packed;
  int pre = block_excl_scan(lane == 0 ? wpacked : 0, sh + 32, &tot_packed);
  pre = __shfl_sync(0xffffffffu, pre, 0);
  const int n_runs = tot_packed >> 16, n_multi = tot_packed & 0xFFFF;
  const int n_single = nseg - n_multi;
  const int n_slots = n_runs - n_single;
  // Runs of multi-run ids are placed from the front of the run list (a run's
  // partial slot has the same index), single runs from the back: the reduce
  // then starts with the ids whose runs must be combined.
  if (tid == 0) {
    sh[81] = n_slots > 0 ? atomicAdd(&hdr[1], n_slots) : 0;
    sh[82] = n_multi > 0 ? atomicAdd(&hdr[3], n_multi) : 0;
    sh[83] = n_single > 0 ? atomicAdd(&hdr[5], n_single) : 0;
    if (nseg > 0) atomicAdd(&hdr[2], nseg);
  }
  __syncthreads();
  const int sbase = sh[81], mbase = sh[82], bbase = sh[83];
  for (int j = 0; j < spw; j += 32) {
    const int sg = warp * spw + j + lane;
    int nr = 0, st = 0, en = 0;
    if (sg < nseg) {
      st = seg[sg];
      en = seg_end(sg);
      nr = (en - st + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    }
    const int pk = sg < nseg ? (nr << 16) | (nr > 1 ? 1 : 0) : 0;
    int incl = pk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int mine = pre + incl - pk;
    pre += __shfl_sync(0xffffffffu, incl, 31);
    if (sg < nseg) {
      const int rb = mine >> 16, mb = mine & 0xFFFF;
      const bool multi = nr > 1;
      const int q0 = rb - (sg - mb);
      const int32_t id = static_cast<int32_t>((src[st] >> tbits) * NB + b);
      for (int k = 0; k < nr; ++k) {
        RunDesc rd;
        rd.start = tbase + st + k * kEmbedBwdChunk;
        rd.end = tbase + min(en, st + (k + 1) * kEmbedBwdChunk);
        rd.id = id;
        rd.slot = multi ? sbase + q0 + k : -1;
        rd.mseg = multi ? mbase + mb : -1;
        rd.nruns = nr;
        rd.first_slot = multi ? sbase + q0 : -1;
        rd.pad = 0;
        runs[multi ? sbase + q0 + k : T - 1 - (bbase + (sg - mb))] = rd;
      }
      if (multi)
        for (int hh = 0; hh < nhm; ++hh) counters[(mbase + mb) * nhm + hh] = 0;
    }
  }
}

// Workspace variant: 64-bit keys (id << 32) | t, any T.
__global__ void __launch_bounds__(kSortThreads, 1)
    embed_sort_kernel(const int64_t* __restrict__ ids, int64_t T, int64_t V_real, int nhm, int32_t* hdr,
                      uint64_t* keys_a, uint64_t* keys_b, int32_t* seg_start, int32_t* tsorted, RunDesc* runs,
                      int32_t* counters) {
  __shared__ int sh_warp[33];
  __shared__ int hist[kRadix];
  __shared__ int carry[kRadix];
  __shared__ int warp_cnt[kSortWarps][kRadix];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Phase 0: stable compaction of the valid ids, key = (id << 32) | t.
  int n = 0;
  for (int64_t base = 0; base < T; base += kSortTile) {
    int cnt = 0;
    int64_t t0 = base + static_cast<int64_t>(tid) * kSortItems;
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      int64_t t = t0 + j;
      if (t < T) {
        int64_t id = ids[t];
        cnt += (id >= 0 && id < V_real) ? 1 : 0;
      }
    }
    int tot;
    int pos = n + block_excl_scan(cnt, sh_warp, &tot);
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      int64_t t = t0 + j;
      if (t < T) {
        int64_t id = ids[t];
        if (id >= 0 && id < V_real) keys_a[pos++] = (static_cast<uint64_t>(id) << 32) | static_cast<uint64_t>(t);
      }
    }
    n += tot;
  }
  __syncthreads();

  // Phase 1: LSD radix passes over the id bits (stable, so t stays ascending).
  int idbits = 1;
  while (idbits < 40 && (int64_t(1) << idbits) < V_real) ++idbits;
  uint64_t* src = keys_a;
  uint64_t* dst = keys_b;
  for (int shift = 0; shift < idbits; shift += 8) {
    const int sh = 32 + shift;
    for (int i = tid; i < kRadix; i += kSortThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kSortThreads) atomicAdd(&hist[(src[i] >> sh) & 0xFF], 1);
    __syncthreads();
    {
      int v = tid < kRadix ? hist[tid] : 0;
      int tot;
      int ex = block_excl_scan(v, sh_warp, &tot);
      if (tid < kRadix) carry[tid] = ex;
    }
    __syncthreads();
    for (int base = 0; base < n; base += kSortTile) {
      for (int i = tid; i < kSortWarps * kRadix; i += kSortThreads) (&warp_cnt[0][0])[i] = 0;
      __syncthreads();
      uint64_t key[kSortItems];
      int dig[kSortItems], rank[kSortItems];
#pragma unroll
      for (int j = 0; j < kSortItems; ++j) {
        const int idx = base + warp * (32 * kSortItems) + j * 32 + lane;   // warp-striped
        const bool ok = idx < n;
        key[j] = ok ? src[idx] : 0ull;
        const int d = ok ? static_cast<int>((key[j] >> sh) & 0xFF) : (kRadix + lane);
        dig[j] = d;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        const int before = __popc(peers & ((1u << lane) - 1u));
        int c0 = 0;
        if (ok) c0 = warp_cnt[warp][d];
        __syncwarp();
        if (ok && before == 0) warp_cnt[warp][d] = c0 + __popc(peers);
        __syncwarp();
        rank[j] = c0 + before;
      }
      __syncthreads();
      if (tid < kRadix) {
        int s = carry[tid];
        for (int w = 0; w < kSortWarps; ++w) {
          int c = warp_cnt[w][tid];
          warp_cnt[w][tid] = s;
          s += c;
        }
        carry[tid] = s;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kSortItems; ++j) {
        const int idx = base + warp * (32 * kSortItems) + j * 32 + lane;
        if (idx < n) dst[warp_cnt[warp][dig[j]] + rank[j]] = key[j];
      }
      __syncthreads();
    }
    uint64_t* tmp = src;
    src = dst;
    dst = tmp;
  }

  // Phase 2a: id boundaries in the sorted keys; sorted token indices.
  int nseg = 0;
  int32_t* seg_ids = reinterpret_cast<int32_t*>(dst);   // the free key buffer
  for (int base = 0; base < n; base += kSortTile) {
    int cnt = 0;
    const int p0 = base + tid * kSortItems;
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      const int q = p0 + j;
      if (q < n) {
        tsorted[q] = static_cast<int32_t>(src[q] & 0xFFFFFFFFull);
        if (q == 0 || (src[q] >> 32) != (src[q - 1] >> 32)) ++cnt;
      }
    }
    int tot;
    int s = nseg + block_excl_scan(cnt, sh_warp, &tot);
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
      const int q = p0 + j;
      if (q < n && (q == 0 || (src[q] >> 32) != (src[q - 1] >> 32))) {
        seg_start[s] = q;
        seg_ids[s] = static_cast<int32_t>(src[q] >> 32);
        ++s;
      }
    }
    nseg += tot;
  }
  __syncthreads();
  auto id_of = [&](int sg) { return static_cast<int>(seg_ids[sg]); };
  auto seg_at = [&](int sg) { return seg_start[sg]; };
  build_runs(seg_at, nseg, n, static_cast<int>(T), (nseg + kSortThreads - 1) / kSortThreads, nhm, id_of, sh_warp, hdr, runs,
             counters);
  if (tid == 0) {
    hdr[0] = n;
    hdr[2] = nseg;
    plan_seal(hdr, static_cast<int>(T), nhm, V_real);
  }
}

// ---------------------------------------------------------------------------
// Backward, step 2: persistent segmented reduction. Work item = (run, column
// slice): 128 threads x 16 bytes for the run of a single-run id, 128 threads x
// 8 bytes for a run of a multi-run id.
// ---------------------------------------------------------------------------
template <typename TE>
__device__ __forceinline__ void widen(const uint4& v, float (&o)[16 / sizeof(TE)]);
template <>
__device__ __forceinline__ void widen<uint16_t>(const uint4& v, float (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void widen<float>(const uint4& v, float (&o)[4]) {
  o[0] = __uint_as_float(v.x);
  o[1] = __uint_as_float(v.y);
  o[2] = __uint_as_float(v.z);
  o[3] = __uint_as_float(v.w);
}

// 8 bytes of dE (four bf16 or two fp32 values), widened.
template <typename TE>
__device__ __forceinline__ void widen(const uint2& v, float (&o)[8 / sizeof(TE)]);
template <>
__device__ __forceinline__ void widen<uint16_t>(const uint2& v, float (&o)[4]) {
  o[0] = __uint_as_float(v.x << 16);
  o[1] = __uint_as_float(v.x & 0xFFFF0000u);
  o[2] = __uint_as_float(v.y << 16);
  o[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void widen<float>(const uint2& v, float (&o)[2]) {
  o[0] = __uint_as_float(v.x);
  o[1] = __uint_as_float(v.y);
}

// acc += dE rows t_p, t_{p+1}, ..., t_{p+N-1} (this thread's 16-byte column
// chunk), the N loads issued before the first add, the adds in token order.
// Token t_j is lane j's my_t. Straight-line code for each N, so a short run
// issues only its own loads and adds.
template <int N, typename TE, bool STREAM, typename LT = uint4>
__device__ __forceinline__ void add_rows(const TE* __restrict__ dE, int64_t H, int col, int my_t, int p, bool active,
                                         float (&acc)[sizeof(LT) / sizeof(TE)]) {
  constexpr int VEC = sizeof(LT) / sizeof(TE);
  LT v[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int t = __shfl_sync(0xffffffffu, my_t, (p + k) & 31);
    v[k] = LT{};
    // With one problem dE is read once: streaming loads (evict first) keep the
    // L2 for the dW rows. The n-gram tables read dE once each, from L2.
    const LT* src = reinterpret_cast<const LT*>(dE + static_cast<int64_t>(t) * H + col);
    if (active) v[k] = STREAM ? __ldcs(src) : __ldg(src);
  }
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float f[VEC];
    widen<TE>(v[k], f);
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = acc[e] + f[e];
  }
}

// Bucketed counting sort: the bucketed variant's CTAs, each sorting its ids by
// q = id / NB with one counting pass instead of radix passes. With nq values
// of q, kCntWarps warps each own a contiguous share of the bucket's keys (in
// token order) and a row of nq counters:
//   1. each warp counts its keys per q (shared-memory atomics; the rows of
//      warps 2k and 2k+1 share 32-bit words, one 16-bit half each);
//   2. per q, the rows become exclusive prefixes across the warps, and a block
//      scan over q gives each q's first sorted position, the runs before it,
//      the ids (non-empty q) before it and the multi-run ids before it;
//   3. each warp places its keys' tokens straight into tsorted, in token order
//      within each q, so the sort is stable;
//   4. the bucket's runs are written in parallel, one thread per run, each
//      finding its q by binary search over the runs-before counts.
// The tokens, runs and run order produced are exactly those of the radix
// variant.
constexpr int kCntWarps = 8;
constexpr size_t kCountSmemBudget = 200 * 1024;

// Keys per segment: with CL > 1, CTA rank r of a cluster loads tokens
// [r * Tc, (r + 1) * Tc) and every CTA keeps one segment of Tc keys per rank.
__host__ __device__ constexpr int count_seg_cap(int T, int CL) {
  return CL == 1 ? T : (((T + CL - 1) / CL + 31) & ~31);
}

// The per-warp counters of q live two warps to a 32-bit word (every count and
// position is below T <= 16384 < 2^16), in rows padded by one word per 32 q so
// that a thread's consecutive q fall in distinct banks across a warp.
__host__ __device__ constexpr int qpad(int q) { return q + (q >> 5); }
__host__ __device__ constexpr int64_t count_row_words(int64_t nq) { return nq + (nq >> 5) + 1; }

size_t count_sort_smem(int64_t T, int64_t nq, int CL) {   // key segments, packed counter rows, three per-q arrays
  return static_cast<size_t>(CL) * count_seg_cap(static_cast<int>(T), CL) * sizeof(uint32_t) +
         static_cast<size_t>(kCntWarps / 2) * count_row_words(nq) * sizeof(uint32_t) +
         static_cast<size_t>(3) * nq * sizeof(int);
}

// Thread-block-cluster helpers for the clustered id load.
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {   // the same smem word in CTA `rank`
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return r;
}
__device__ __forceinline__ void cl_store(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// ROUNDS: rounds of 32 tokens per warp in phase A, so that a smaller batch
// does not issue the larger one's predicated rounds.
//
// CL: CTAs per thread-block cluster. With CL == 1 every CTA loads all T ids and
// keeps its own bucket's keys. With CL > 1 the cluster's CTAs own CL
// consecutive buckets and share the loading: rank r loads tokens
// [r * Tc, (r + 1) * Tc) and stores each key of the cluster's buckets into the
// owning CTA's segment r, through distributed shared memory, so the ids cross
// L2 once per cluster instead of once per CTA. Segment r then holds bucket
// keys in token order, and segments follow token order too. The counting
// warps take the segments in order (kCntWarps / CL warps each), which keeps
// the sort stable exactly as with one contiguous key array.
//
// One launch sorts up to three problems of the same T side by side (the
// n-gram backward's tables): blocks [k * nb, (k + 1) * nb) sort problem k into
// nb buckets, nb a multiple of CL so that a cluster stays within one problem.
constexpr int kMaxSortJobs = 3;
struct SortJobs {
  const int64_t* ids[kMaxSortJobs];
  int64_t V_real[kMaxSortJobs];
  int nq[kMaxSortJobs];   // ceil(V_real / nb)
  int32_t* hdr[kMaxSortJobs];
  int32_t* tsorted[kMaxSortJobs];
  RunDesc* runs[kMaxSortJobs];
  int32_t* counters[kMaxSortJobs];
  int nb;                 // buckets per problem
};

template <int ROUNDS, int CL>
__global__ void __launch_bounds__(kBktThreads, 1)
    embed_sort_count_kernel(const __grid_constant__ SortJobs J, int T, int tbits, int nhm, uint32_t nb_magic) {
  static_assert(CL >= 1 && CL <= 8 && kCntWarps % CL == 0, "counting warps split evenly over the segments");
  const int job = static_cast<int>(blockIdx.x) / J.nb;   // the same for every CTA of a cluster
  const int64_t* __restrict__ ids = job == 2 ? J.ids[2] : (job == 1 ? J.ids[1] : J.ids[0]);
  const int64_t V_real = job == 2 ? J.V_real[2] : (job == 1 ? J.V_real[1] : J.V_real[0]);
  const int nq = job == 2 ? J.nq[2] : (job == 1 ? J.nq[1] : J.nq[0]);
  int32_t* hdr = job == 2 ? J.hdr[2] : (job == 1 ? J.hdr[1] : J.hdr[0]);
  int32_t* tsorted = job == 2 ? J.tsorted[2] : (job == 1 ? J.tsorted[1] : J.tsorted[0]);
  RunDesc* runs = job == 2 ? J.runs[2] : (job == 1 ? J.runs[1] : J.runs[0]);
  int32_t* counters = job == 2 ? J.counters[2] : (job == 1 ? J.counters[1] : J.counters[0]);
  extern __shared__ __align__(16) uint32_t csm[];
  const int Tc = count_seg_cap(T, CL);
  uint32_t* ka = csm;                                  // [CL][Tc] this bucket's keys, token order
  const int nqp = static_cast<int>(count_row_words(nq));
  uint32_t* rows = csm + CL * Tc;                      // [kCntWarps / 2][nqp] warps 2k, 2k+1 in halves of word k
  int* bstart = reinterpret_cast<int*>(rows + (kCntWarps / 2) * nqp);   // [nq] first sorted position of q (its count, in step 2)
  int* brun = bstart + nq;                             // [nq] runs before q
  int* bseg = brun + nq;                               // [nq] ids before q | multi-run ids before q << 16
  __shared__ int sh[96];
  __shared__ uint64_t sh64[33];
  __shared__ int segn[CL];                             // keys in each segment
  __shared__ int wdc[CL > 1 ? kBktWarps * CL : 1];     // per warp and destination rank: keys sent
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const uint32_t NB = static_cast<uint32_t>(J.nb), b = blockIdx.x - static_cast<uint32_t>(job * J.nb);

  grid_dep_launch();   // the reduce may be scheduled from here on; it waits for this grid to end

  int m = 0;
  if constexpr (CL == 1) {
    // Phase A, as in the radix variant: every id loaded before any is used.
    const int tpw = ((T + kBktWarps - 1) / kBktWarps + 31) & ~31;
    int64_t idv[ROUNDS];
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const int t = warp * tpw + j * 32 + lane;
      idv[j] = (j * 32 < tpw && t < T) ? __ldg(ids + t) : -1;
    }
    for (int i = tid; i < (kCntWarps / 2) * nqp; i += kBktThreads) rows[i] = 0;   // while the loads are in flight
    uint32_t tkey[ROUNDS];
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      uint32_t k = 0xFFFFFFFFu;
      if (idv[j] >= 0 && idv[j] < V_real) {
        const uint32_t u = static_cast<uint32_t>(idv[j]);
        const uint32_t q = __umulhi(u, nb_magic);   // u / NB, exact for u < 2^32 / NB
        if (u - q * NB == b) k = (q << tbits) | static_cast<uint32_t>(warp * tpw + j * 32 + lane);
      }
      tkey[j] = k;
    }
    int wcount = 0;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) wcount += __popc(__ballot_sync(0xffffffffu, tkey[j] != 0xFFFFFFFFu));
    if (lane == 0) sh[warp] = wcount;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < kBktWarps; ++w) {
      const int c = sh[w];
      wbase += w < warp ? c : 0;
      m += c;
    }
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const bool ok = tkey[j] != 0xFFFFFFFFu;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      if (ok) ka[wbase + __popc(bal & lt_mask)] = tkey[j];
      wbase += __popc(bal);
    }
    if (tid == 0) segn[0] = m;
  } else {
    // Phase A, clustered. The arrive marks this CTA as started; the wait
    // before the first remote store makes sure every CTA of the cluster is.
    cl_arrive_relaxed();
    const uint32_t rank = cl_rank(), cbase = b - rank;
    const int t_lo = static_cast<int>(rank) * Tc, t_hi = min(T, t_lo + Tc);
    const int tpw = ((Tc + kBktWarps - 1) / kBktWarps + 31) & ~31;
    int64_t idv[ROUNDS];
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const int t = t_lo + warp * tpw + j * 32 + lane;
      idv[j] = (j * 32 < tpw && t < t_hi) ? __ldg(ids + t) : -1;
    }
    for (int i = tid; i < (kCntWarps / 2) * nqp; i += kBktThreads) rows[i] = 0;   // while the loads are in flight
    uint32_t tkey[ROUNDS];
    int dst[ROUNDS], lpos[ROUNDS];
    int sent = 0;   // lane d < CL: this warp's keys for rank d so far
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      uint32_t k = 0;
      int d = CL;   // CL: not a bucket of this cluster
      if (idv[j] >= 0 && idv[j] < V_real) {
        const uint32_t u = static_cast<uint32_t>(idv[j]);
        const uint32_t q = __umulhi(u, nb_magic);   // u / NB, exact for u < 2^32 / NB
        const uint32_t r = u - q * NB - cbase;      // wraps above CL for buckets before this cluster's
        if (r < static_cast<uint32_t>(CL)) {
          d = static_cast<int>(r);
          k = (q << tbits) | static_cast<uint32_t>(t_lo + warp * tpw + j * 32 + lane);
        }
      }
      int lp = 0, add = 0;
#pragma unroll
      for (int dd = 0; dd < CL; ++dd) {
        const unsigned bal = __ballot_sync(0xffffffffu, d == dd);
        if (d == dd) lp = __popc(bal & lt_mask);
        if (lane == dd) add = __popc(bal);
      }
      lpos[j] = __shfl_sync(0xffffffffu, sent, d < CL ? d : 0) + lp;
      sent += add;
      tkey[j] = k;
      dst[j] = d;
    }
    if (lane < CL) wdc[warp * CL + lane] = sent;
    __syncthreads();
    int wpre = 0, tot = 0;   // lane d < CL: keys for rank d from the warps before this one, and from all
    if (lane < CL)
      for (int w = 0; w < kBktWarps; ++w) {
        const int c = wdc[w * CL + lane];
        wpre += w < warp ? c : 0;
        tot += c;
      }
    cl_wait();   // every CTA of the cluster has started
    if (warp == 0 && lane < CL) cl_store(cl_map(&segn[rank], lane), static_cast<uint32_t>(tot));
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const int base = __shfl_sync(0xffffffffu, wpre, dst[j] < CL ? dst[j] : 0);
      if (dst[j] < CL) cl_store(cl_map(&ka[static_cast<int>(rank) * Tc + base + lpos[j]], dst[j]), tkey[j]);
    }
    cl_arrive();   // the stores above are visible cluster-wide after the wait
    cl_wait();
#pragma unroll
    for (int r = 0; r < CL; ++r) m += segn[r];
  }
  // This bucket's place in tsorted; the header is zeroed by the kernel before
  // this one. The claim's result is first needed in step 3.
  grid_dep_wait();
  int tb = 0;
  if (tid == 0 && m > 0) tb = atomicAdd(&hdr[0], m);
  if (tid == 0 && b == 0) plan_seal(hdr, T, nhm, V_real);
  __syncthreads();

  // Counting warp w takes part w % (kCntWarps / CL) of segment w / (kCntWarps / CL).
  constexpr int kSpw = kCntWarps / CL;
  int k_lo = 0, k_hi = 0;
  const uint32_t* kseg = ka;
  if (warp < kCntWarps) {
    const int sgi = warp / kSpw, scnt = segn[sgi];
    const int share = ((scnt + kSpw - 1) / kSpw + 31) & ~31;   // whole rounds
    k_lo = min((warp % kSpw) * share, scnt);
    k_hi = min(k_lo + share, scnt);
    kseg = ka + sgi * Tc;
  }

  // Step 1: per-warp counts of each q, by shared-memory atomics (the counts do
  // not depend on the order of the additions).
  uint32_t* const row = rows + ((warp % kCntWarps) >> 1) * nqp;   // used by the counting warps only
  const uint32_t half = 16u * static_cast<uint32_t>(warp & 1);
  if (warp < kCntWarps)
    for (int i = k_lo + lane; i < k_hi; i += 32) atomicAdd(&row[qpad(static_cast<int>(kseg[i] >> tbits))], 1u << half);
  __syncthreads();

  // Step 2: thread tid owns the q in [q0, q1). Rows become exclusive prefixes
  // across the warps; the four per-q counts are scanned packed 16 bits each
  // (every total is at most T <= 16384).
  const int bpt = (nq + kBktThreads - 1) / kBktThreads;
  const int q0 = min(tid * bpt, nq), q1 = min(q0 + bpt, nq);
  uint64_t mine = 0;
  for (int q = q0; q < q1; ++q) {
    const int qi = qpad(q);
    int run = 0;
#pragma unroll
    for (int k = 0; k < kCntWarps / 2; ++k) {
      const uint32_t v = rows[k * nqp + qi];
      const int c0 = static_cast<int>(v & 0xFFFFu), c1 = static_cast<int>(v >> 16);
      rows[k * nqp + qi] = static_cast<uint32_t>(run) | (static_cast<uint32_t>(run + c0) << 16);
      run += c0 + c1;
    }
    bstart[q] = run;
    const int nr = (run + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    mine += static_cast<uint64_t>(run) | (static_cast<uint64_t>(nr) << 16) |
            (static_cast<uint64_t>(run > 0) << 32) | (static_cast<uint64_t>(nr > 1) << 48);
  }
  uint64_t tot;
  uint64_t pre = block_excl_scan64(mine, sh64, &tot);
  for (int q = q0; q < q1; ++q) {
    const int cnt = bstart[q];
    const int p_cnt = static_cast<int>(pre & 0xFFFF), p_run = static_cast<int>((pre >> 16) & 0xFFFF);
    const int p_seg = static_cast<int>((pre >> 32) & 0xFFFF), p_multi = static_cast<int>(pre >> 48);
    bstart[q] = p_cnt;
    brun[q] = p_run;
    bseg[q] = p_seg | (p_multi << 16);
    const int qi = qpad(q);
#pragma unroll
    for (int k = 0; k < kCntWarps / 2; ++k) rows[k * nqp + qi] += static_cast<uint32_t>(p_cnt) * 0x10001u;
    const int nr = (cnt + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    pre += static_cast<uint64_t>(cnt) | (static_cast<uint64_t>(nr) << 16) | (static_cast<uint64_t>(cnt > 0) << 32) |
           (static_cast<uint64_t>(nr > 1) << 48);
  }
  const int n_runs = static_cast<int>((tot >> 16) & 0xFFFF);
  const int nseg = static_cast<int>((tot >> 32) & 0xFFFF), n_multi = static_cast<int>(tot >> 48);
  const int n_single = nseg - n_multi, n_slots = n_runs - n_single;
  // Runs of multi-run ids go to the front of the run list (a run's partial
  // slot has the same index), single runs to its back, as in the radix variant.
  int c_slot = 0, c_multi = 0, c_single = 0;
  if (tid == 0) {
    sh[80] = tb;
    c_slot = n_slots > 0 ? atomicAdd(&hdr[1], n_slots) : 0;
    c_multi = n_multi > 0 ? atomicAdd(&hdr[3], n_multi) : 0;
    c_single = n_single > 0 ? atomicAdd(&hdr[5], n_single) : 0;
    if (nseg > 0) atomicAdd(&hdr[2], nseg);
  }
  __syncthreads();
  const int tbase = sh[80];
  const uint32_t tmask = (1u << tbits) - 1u;

  // Step 3: tokens into place.
  if (warp < kCntWarps) {
    for (int j = k_lo; j < k_hi; j += 32) {
      const int i = j + lane;
      const bool ok = i < k_hi;
      const uint32_t key = ok ? kseg[i] : 0u;
      const uint32_t q = ok ? key >> tbits : 0xFFFFFFFFu;
      const uint32_t peers = __match_any_sync(0xffffffffu, q);
      int base = 0;
      if (ok) base = static_cast<int>((row[qpad(static_cast<int>(q))] >> half) & 0xFFFFu);
      __syncwarp();
      if (ok) {
        tsorted[tbase + base + __popc(peers & lt_mask)] = static_cast<int32_t>(key & tmask);
        if (lane == __ffs(peers) - 1)   // the other half belongs to warp w ^ 1
          atomicAdd(&row[qpad(static_cast<int>(q))], static_cast<uint32_t>(__popc(peers)) << half);
      }
      __syncwarp();
    }
  }
  if (tid == 0) {
    sh[81] = c_slot;
    sh[82] = c_multi;
    sh[83] = c_single;
  }
  __syncthreads();
  const int sbase = sh[81], mbase = sh[82], bbase = sh[83];

  // Step 4: the runs, one thread each.
  for (int r = tid; r < n_runs; r += kBktThreads) {
    int lo = 0, hi = nq - 1;   // the largest q with brun[q] <= r is the run's (non-empty) q
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (brun[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int q = lo;
    const int st = bstart[q];
    const int cnt = (q + 1 < nq ? bstart[q + 1] : m) - st;
    const int nr = (cnt + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    const int k = r - brun[q];
    const int p_seg = bseg[q] & 0xFFFF, p_multi = bseg[q] >> 16;
    const bool multi = nr > 1;
    const int first = brun[q] - (p_seg - p_multi);   // slots of the multi-run ids before q
    RunDesc rd;
    rd.start = tbase + st + k * kEmbedBwdChunk;
    rd.end = tbase + st + min(cnt, (k + 1) * kEmbedBwdChunk);
    rd.id = static_cast<int32_t>(static_cast<uint32_t>(q) * NB + b);
    rd.slot = multi ? sbase + first + k : -1;
    rd.mseg = multi ? mbase + p_multi : -1;
    rd.nruns = nr;
    rd.first_slot = multi ? sbase + first : -1;
    rd.pad = 0;
    runs[multi ? sbase + first + k : T - 1 - (bbase + (p_seg - p_multi))] = rd;
    if (multi && k == 0)
      for (int hh = 0; hh < nhm; ++hh) counters[(mbase + p_multi) * nhm + hh] = 0;
  }
}

// One sorted problem for the reduce: its workspace arrays and its dW. The
// n-gram backward reduces three (the token table and two n-gram tables) in one
// launch, their items numbered one problem after the other.
struct EmbSlot {
  int32_t* hdr;
  int32_t rows;   // V_real of the problem: the plan must index the same rows
  const int32_t* tsorted;
  const RunDesc* runs;
  float* dW;
  float* partials;
  int32_t* counters;
};
constexpr int kMaxSlots = 3;
struct EmbSlots {
  EmbSlot s[kMaxSlots];
  int n;
};

// PV consecutive fp32 values of a row (16-byte aligned for PV >= 4, 8-byte for
// PV = 2), loaded and stored as vectors; cg = at L2.
template <int PV>
struct FRow;
template <>
struct FRow<4> {
  __device__ static void ld_cg(const float* p, float (&o)[4]) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  }
  __device__ static void ld(const float* p, float (&o)[4]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  }
  __device__ static void st_cg(float* p, const float (&o)[4]) {
    __stcg(reinterpret_cast<float4*>(p), make_float4(o[0], o[1], o[2], o[3]));
  }
  __device__ static void st(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <>
struct FRow<2> {
  __device__ static void ld_cg(const float* p, float (&o)[2]) {
    const float2 a = __ldcg(reinterpret_cast<const float2*>(p));
    o[0] = a.x; o[1] = a.y;
  }
  __device__ static void ld(const float* p, float (&o)[2]) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    o[0] = a.x; o[1] = a.y;
  }
  __device__ static void st_cg(float* p, const float (&o)[2]) { __stcg(reinterpret_cast<float2*>(p), make_float2(o[0], o[1])); }
  __device__ static void st(float* p, const float (&o)[2]) { *reinterpret_cast<float2*>(p) = make_float2(o[0], o[1]); }
};

// The end of one run of a multi-run id over one column slice, its sum in
// token order in hand (PV values per thread): the sum goes to the run's
// partial slot; the last of the id's runs to finish then adds the id's run
// sums left to right into its dW row, loading kAhead of them at a time so that
// a hot id's combine waits for about nruns / kAhead round trips, not nruns.
template <int PV, int kAhead>
__device__ __forceinline__ void multi_run_finish(const float (&acc)[PV], int H, int col, bool active,
                                                 const RunDesc& rd, float* __restrict__ dW, float* partials,
                                                 int32_t* ctr, int* s_last) {
  if (active) FRow<PV>::st_cg(partials + static_cast<int64_t>(rd.slot) * H + col, acc);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(ctr, 1);
    *s_last = (prev == rd.nruns - 1) ? 1 : 0;
    if (*s_last) *ctr = 0;   // every run is in: back to the plan's zero
    __threadfence();
  }
  __syncthreads();
  if (*s_last && active) {
    float tot[PV];
    FRow<PV>::ld_cg(partials + static_cast<int64_t>(rd.first_slot) * H + col, tot);
    for (int j0 = 1; j0 < rd.nruns; j0 += kAhead) {
      float a[kAhead][PV];
#pragma unroll
      for (int k = 0; k < kAhead; ++k) {
        const int j = min(j0 + k, rd.nruns - 1);   // past the end: a valid slot, not added
        FRow<PV>::ld_cg(partials + static_cast<int64_t>(rd.first_slot + j) * H + col, a[k]);
      }
#pragma unroll
      for (int k = 0; k < kAhead; ++k)
        if (j0 + k < rd.nruns) {
#pragma unroll
          for (int e = 0; e < PV; ++e) tot[e] = tot[e] + a[k][e];
        }
    }
    float* row = dW + static_cast<int64_t>(rd.id) * H + col;
    float w[PV];
    FRow<PV>::ld(row, w);
#pragma unroll
    for (int e = 0; e < PV; ++e) w[e] = w[e] + tot[e];
    FRow<PV>::st(row, w);
  }
}

// A narrow item: one run of a multi-run id over half a wide slice's columns,
// 8 bytes of dE per thread. A multi-run id's runs hold 32 tokens (all but its
// last), and its last run to finish combines all of its run sums: both steps
// wait on loads in flight. In the registers of a wide item (16 bytes per
// thread, 8 rows and 4 run sums ahead), a narrow one keeps 16 rows and 8 run
// sums ahead: the hottest id of a Zipf batch (35 runs at 8192 tokens) waits
// for 2 rounds of row loads instead of 4 and 5 rounds of run sums instead of
// 9, at the price of twice as many items for the multi-run ids. The additions
// and their order are those of a wide item.
template <typename TE, bool STREAM>
__device__ __forceinline__ void reduce_multi_run_narrow(const TE* __restrict__ dE, int H, int col, bool active,
                                                        const RunDesc& rd, int my_t, float* __restrict__ dW,
                                                        float* partials, int32_t* ctr, int* s_last) {
  constexpr int PV = 8 / sizeof(TE);
  constexpr int U = 16;   // rows loaded ahead of the sequential adds
  const int len = rd.end - rd.start;   // <= 32
  float acc[PV];
#pragma unroll
  for (int e = 0; e < PV; ++e) acc[e] = 0.0f;
  for (int p = 0; p < len; p += U) {   // tokens in ascending t, one add each
    switch (len - p < U ? len - p : U) {
      case 1: add_rows<1, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 2: add_rows<2, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 3: add_rows<3, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 4: add_rows<4, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 5: add_rows<5, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 6: add_rows<6, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 7: add_rows<7, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 8: add_rows<8, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 9: add_rows<9, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 10: add_rows<10, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 11: add_rows<11, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 12: add_rows<12, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 13: add_rows<13, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 14: add_rows<14, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      case 15: add_rows<15, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
      default: add_rows<U, TE, STREAM, uint2>(dE, H, col, my_t, p, active, acc); break;
    }
  }
  multi_run_finish<PV, 8>(acc, H, col, active, rd, dW, partials, ctr, s_last);
}

// STREAM: dE is read once (one problem), with evict-first loads.
template <typename TE, bool STREAM>
__global__ void __launch_bounds__(128)
    embed_reduce_kernel(const __grid_constant__ EmbSlots sl, const TE* __restrict__ dE, int H, int nh,
                        uint32_t nh_magic, int cap, int32_t* status) {
  constexpr int VEC = 16 / sizeof(TE);
  constexpr int NQ = VEC / 4;
  constexpr int U = 8;               // rows loaded ahead of the sequential adds
  constexpr int kCombineAhead = 4;   // run sums loaded ahead in a combine
  __shared__ int s_last;
  __shared__ int s_next[2];
  const int lane = threadIdx.x & 31;
  grid_dep_wait();   // the sorts' headers, runs and tokens
  // Every problem must hold a plan made for this shape (T = cap, the same
  // column slices and rows); otherwise nothing is added and the call reports
  // VCE_ERR_ARG.
  bool planned = true;
  for (int k = 0; k < sl.n; ++k)
    planned = planned && sl.s[k].hdr[kHdrPlanMark] == kPlanMark && sl.s[k].hdr[kHdrPlanT] == cap &&
              sl.s[k].hdr[kHdrPlanNh] == nh && sl.s[k].hdr[kHdrPlanRows] == sl.s[k].rows;
  if (!planned) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    return;
  }
  // In each problem, runs [0, n_front) sit at the front of the list, the other
  // n_back at its end (indices cap-1, cap-2, ...). Problem k's items are
  // [base_k, base_k+1).
  const int nf0 = sl.s[0].hdr[1];
  const int nf1 = sl.n > 1 ? sl.s[1].hdr[1] : 0;
  const int nf2 = sl.n > 2 ? sl.s[2].hdr[1] : 0;
  const int base1 = (nf0 + sl.s[0].hdr[5]) * nh;
  const int base2 = base1 + (sl.n > 1 ? (nf1 + sl.s[1].hdr[5]) * nh : 0);
  const int n_items = base2 + (sl.n > 2 ? (nf2 + sl.s[2].hdr[5]) * nh : 0);
  // Items are handed out in order: the first one per CTA by its index, the
  // rest from a counter in the first problem's header (zeroed before this
  // kernel), claimed one item ahead so that the claim's round trip overlaps
  // the current item.
  int32_t* item_ctr = sl.s[0].hdr + kHdrItem;
  int it = 0;
  for (int item = blockIdx.x; item < n_items; ++it) {
    int next = 0;
    if (threadIdx.x == 0) {
      // One claim per item in all: the claim that draws n_items - 1 is the
      // last one, and puts the counter back to zero for the plan's next use.
      const int prev = atomicAdd(item_ctr, 1);
      if (prev == n_items - 1) atomicExch(item_ctr, 0);
      next = prev + static_cast<int>(gridDim.x);
    }
    // this item's problem (a uniform choice among at most three)
    const int k = item >= base2 ? 2 : (item >= base1 ? 1 : 0);
    const int li = item - (k == 2 ? base2 : (k == 1 ? base1 : 0));
    const int n_front = k == 2 ? nf2 : (k == 1 ? nf1 : nf0);
    const RunDesc* __restrict__ runs = k == 2 ? sl.s[2].runs : (k == 1 ? sl.s[1].runs : sl.s[0].runs);
    const int32_t* __restrict__ tsorted = k == 2 ? sl.s[2].tsorted : (k == 1 ? sl.s[1].tsorted : sl.s[0].tsorted);
    float* __restrict__ dW = k == 2 ? sl.s[2].dW : (k == 1 ? sl.s[1].dW : sl.s[0].dW);
    float* partials = k == 2 ? sl.s[2].partials : (k == 1 ? sl.s[1].partials : sl.s[0].partials);
    int32_t* counters = k == 2 ? sl.s[2].counters : (k == 1 ? sl.s[1].counters : sl.s[0].counters);
    // li / nh by a multiply-high when the host found it exact for every item
    const int r = nh_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(li), nh_magic)) : li / nh;
    const int hs = li - r * nh;
    const RunDesc rd = runs[r < n_front ? r : cap - 1 - (r - n_front)];
    const int len = rd.end - rd.start;   // <= 32
    const int col = hs * 128 * VEC + static_cast<int>(threadIdx.x) * VEC;
    const bool active = col < H;
    // the run's token indices, one per lane, broadcast below
    const int my_t = lane < len ? tsorted[rd.start + lane] : 0;
    float4* row = reinterpret_cast<float4*>(dW + static_cast<int64_t>(rd.id) * H + col);
    float4 w[NQ];
    if (rd.slot < 0 && active) {   // single-run id: fetch the row now, add once the sum is ready
#pragma unroll
      for (int q = 0; q < NQ; ++q) w[q] = __ldcg(row + q);   // at L2: the row is not read again here
    }
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
    for (int p = 0; p < len; p += U) {   // tokens in ascending t, one add each
      switch (len - p < U ? len - p : U) {
        case 1: add_rows<1, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        case 2: add_rows<2, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        case 3: add_rows<3, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        case 4: add_rows<4, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        case 5: add_rows<5, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        case 6: add_rows<6, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        case 7: add_rows<7, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        default: add_rows<U, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
      }
    }
    if (rd.slot < 0) {
      if (active) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          w[q].x = w[q].x + acc[4 * q + 0];
          w[q].y = w[q].y + acc[4 * q + 1];
          w[q].z = w[q].z + acc[4 * q + 2];
          w[q].w = w[q].w + acc[4 * q + 3];
          row[q] = w[q];
        }
      }
    } else {
      if (active) {
        float4* slot = reinterpret_cast<float4*>(partials + static_cast<int64_t>(rd.slot) * H + col);
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          __stcg(slot + q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) {
        const int prev = atomicAdd(&counters[rd.mseg * nh + hs], 1);
        s_last = (prev == rd.nruns - 1) ? 1 : 0;
        if (s_last) counters[rd.mseg * nh + hs] = 0;   // every run is in: back to the plan's zero
        __threadfence();
      }
      __syncthreads();
      if (s_last && active) {
        // Last run of this id to finish: add the run sums left to right.
        float tot[VEC];
        const float4* s0 = reinterpret_cast<const float4*>(partials + static_cast<int64_t>(rd.first_slot) * H + col);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float4 a = __ldcg(s0 + q);
          tot[4 * q] = a.x; tot[4 * q + 1] = a.y; tot[4 * q + 2] = a.z; tot[4 * q + 3] = a.w;
        }
        // Run sums are loaded kCombineAhead at a time, so a hot id's combine
        // waits for about nruns / kCombineAhead round trips, not nruns.
        for (int j0 = 1; j0 < rd.nruns; j0 += kCombineAhead) {
          float4 a[kCombineAhead][NQ];
#pragma unroll
          for (int k = 0; k < kCombineAhead; ++k) {
            const int j = min(j0 + k, rd.nruns - 1);   // past the end: a valid slot, not added
            const float4* sj =
                reinterpret_cast<const float4*>(partials + static_cast<int64_t>(rd.first_slot + j) * H + col);
#pragma unroll
            for (int q = 0; q < NQ; ++q) a[k][q] = __ldcg(sj + q);
          }
#pragma unroll
          for (int k = 0; k < kCombineAhead; ++k) {
            if (j0 + k < rd.nruns) {   // left to right
#pragma unroll
              for (int q = 0; q < NQ; ++q) {
                tot[4 * q] = tot[4 * q] + a[k][q].x;
                tot[4 * q + 1] = tot[4 * q + 1] + a[k][q].y;
                tot[4 * q + 2] = tot[4 * q + 2] + a[k][q].z;
                tot[4 * q + 3] = tot[4 * q + 3] + a[k][q].w;
              }
            }
          }
        }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float4 x = row[q];
          x.x = x.x + tot[4 * q + 0];
          x.y = x.y + tot[4 * q + 1];
          x.z = x.z + tot[4 * q + 2];
          x.w = x.w + tot[4 * q + 3];
          row[q] = x;
        }
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) s_next[it & 1] = next;
    __syncthreads();
    item = s_next[it & 1];
  }
}


// The reduce with narrow items for the multi-run ids (reduce_multi_run_narrow).
// Items of problem k: first the runs of its multi-run ids (the front of its
// run list), each in nhf narrow column slices, then its single runs (the back
// of the list), each in nh wide slices, as in embed_reduce_kernel.
template <typename TE, bool STREAM>
__global__ void __launch_bounds__(128, 8)   // eight resident CTAs per SM: at most 64 registers
    embed_reduce_narrow_kernel(const __grid_constant__ EmbSlots sl, const TE* __restrict__ dE, int H, int nh,
                               uint32_t nh_magic, int nhf, uint32_t nhf_magic, int cap, int32_t* status) {
  constexpr int VEC = 16 / sizeof(TE);
  constexpr int NQ = VEC / 4;
  constexpr int U = 8;   // rows loaded ahead of the sequential adds
  __shared__ int s_last;
  __shared__ int s_next[2];
  const int lane = threadIdx.x & 31;
  grid_dep_wait();   // the sorts' headers, runs and tokens
  // Every problem must hold a plan made for this shape (T = cap, the same
  // column slices of multi-run ids and rows); otherwise nothing is added and
  // the call reports VCE_ERR_ARG.
  bool planned = true;
  for (int k = 0; k < sl.n; ++k)
    planned = planned && sl.s[k].hdr[kHdrPlanMark] == kPlanMark && sl.s[k].hdr[kHdrPlanT] == cap &&
              sl.s[k].hdr[kHdrPlanNh] == nhf && sl.s[k].hdr[kHdrPlanRows] == sl.s[k].rows;
  if (!planned) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    return;
  }
  // In each problem, runs [0, n_front) sit at the front of the list, the other
  // n_back at its end (indices cap-1, cap-2, ...). Problem k's items are
  // [base_k, base_k+1).
  const int nf0 = sl.s[0].hdr[1];
  const int nf1 = sl.n > 1 ? sl.s[1].hdr[1] : 0;
  const int nf2 = sl.n > 2 ? sl.s[2].hdr[1] : 0;
  const int base1 = nf0 * nhf + sl.s[0].hdr[5] * nh;
  const int base2 = base1 + (sl.n > 1 ? nf1 * nhf + sl.s[1].hdr[5] * nh : 0);
  const int n_items = base2 + (sl.n > 2 ? nf2 * nhf + sl.s[2].hdr[5] * nh : 0);
  // Items are handed out in order: the first one per CTA by its index, the
  // rest from a counter in the first problem's header (zeroed before this
  // kernel), claimed one item ahead so that the claim's round trip overlaps
  // the current item.
  int32_t* item_ctr = sl.s[0].hdr + kHdrItem;
  int it = 0;
  for (int item = blockIdx.x; item < n_items; ++it) {
    int next = 0;
    if (threadIdx.x == 0) {
      // One claim per item in all: the claim that draws n_items - 1 is the
      // last one, and puts the counter back to zero for the plan's next use.
      const int prev = atomicAdd(item_ctr, 1);
      if (prev == n_items - 1) atomicExch(item_ctr, 0);
      next = prev + static_cast<int>(gridDim.x);
    }
    // this item's problem (a uniform choice among at most three)
    const int k = item >= base2 ? 2 : (item >= base1 ? 1 : 0);
    const int li = item - (k == 2 ? base2 : (k == 1 ? base1 : 0));
    const int n_front = k == 2 ? nf2 : (k == 1 ? nf1 : nf0);
    const RunDesc* __restrict__ runs = k == 2 ? sl.s[2].runs : (k == 1 ? sl.s[1].runs : sl.s[0].runs);
    const int32_t* __restrict__ tsorted = k == 2 ? sl.s[2].tsorted : (k == 1 ? sl.s[1].tsorted : sl.s[0].tsorted);
    float* __restrict__ dW = k == 2 ? sl.s[2].dW : (k == 1 ? sl.s[1].dW : sl.s[0].dW);
    // li / nhf and li / nh by a multiply-high when the host found it exact for
    // every item
    const int n_fi = n_front * nhf;
    const bool front = li < n_fi;
    int r, hs;
    if (front) {
      r = nhf_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(li), nhf_magic)) : li / nhf;
      hs = li - r * nhf;
    } else {
      const int lw = li - n_fi;
      const int rb = nh_magic ? static_cast<int>(__umulhi(static_cast<uint32_t>(lw), nh_magic)) : lw / nh;
      hs = lw - rb * nh;
      r = n_front + rb;
    }
    const RunDesc rd = runs[r < n_front ? r : cap - 1 - (r - n_front)];
    const int len = rd.end - rd.start;   // <= 32
    // the run's token indices, one per lane, broadcast below
    const int my_t = lane < len ? tsorted[rd.start + lane] : 0;
    if (front && (rd.slot < 0 || rd.mseg < 0)) {
      // Only multi-run ids' runs sit at the front of a plan's list.
      if (threadIdx.x == 0 && status) atomicCAS(status, 0, static_cast<int>(VCE_ERR_ARG));
    } else if (front) {
      float* partials = k == 2 ? sl.s[2].partials : (k == 1 ? sl.s[1].partials : sl.s[0].partials);
      int32_t* ctr = (k == 2 ? sl.s[2].counters : (k == 1 ? sl.s[1].counters : sl.s[0].counters)) + rd.mseg * nhf + hs;
      const int col = hs * 64 * VEC + static_cast<int>(threadIdx.x) * (VEC / 2);
      reduce_multi_run_narrow<TE, STREAM>(dE, H, col, col < H, rd, my_t, dW, partials, ctr, &s_last);
    } else {
      // A single-run id: its sum is added straight into its dW row.
      const int col = hs * 128 * VEC + static_cast<int>(threadIdx.x) * VEC;
      const bool active = col < H;
      float4* row = reinterpret_cast<float4*>(dW + static_cast<int64_t>(rd.id) * H + col);
      float4 w[NQ];
      if (active) {   // fetch the row now, add once the sum is ready
#pragma unroll
        for (int q = 0; q < NQ; ++q) w[q] = __ldcg(row + q);   // at L2: the row is not read again here
      }
      float acc[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
      for (int p = 0; p < len; p += U) {   // tokens in ascending t, one add each
        switch (len - p < U ? len - p : U) {
          case 1: add_rows<1, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          case 2: add_rows<2, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          case 3: add_rows<3, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          case 4: add_rows<4, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          case 5: add_rows<5, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          case 6: add_rows<6, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          case 7: add_rows<7, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
          default: add_rows<U, TE, STREAM>(dE, H, col, my_t, p, active, acc); break;
        }
      }
      if (active) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          w[q].x = w[q].x + acc[4 * q + 0];
          w[q].y = w[q].y + acc[4 * q + 1];
          w[q].z = w[q].z + acc[4 * q + 2];
          w[q].w = w[q].w + acc[4 * q + 3];
          row[q] = w[q];
        }
      }
    }
    if (threadIdx.x == 0) s_next[it & 1] = next;
    __syncthreads();
    item = s_next[it & 1];
  }
}

}  // namespace

cudaError_t launch_embed_fwd(const vce_problem& p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                             int32_t* local, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const int esize = p.dtype == VCE_BF16 ? 2 : 4;
  const int row_vecs = static_cast<int>(p.H * esize / 16);
  const int64_t blocks = ceil_div(p.T, kGatherWarps);
  embed_gather_kernel<false><<<static_cast<unsigned>(blocks), kGatherWarps * 32, 0, st>>>(
      ids, static_cast<const uint4*>(W), static_cast<uint4*>(E), owner, local, p.T, p.Vp, p.V_real, p.S,
      row_vecs);
  note_launch(VCE_K_EMBED_GATHER, st);
  return cudaGetLastError();
}

namespace {
cudaError_t plan_multi(const vce_problem* ps, const int64_t* const* ids, void* const* ws, int n, int max_nb,
                       cudaStream_t st);
}  // namespace

// Beside the lookup, a sort without clusters (T <= 8192) takes at most 64 SMs:
// its 1024-thread CTAs hold nearly all of an SM's registers, so each SM it
// takes runs no lookup rows until it exits (measured on GB300, 8192 x 2048
// Qwen3-like ids: the lookup with the plan 18.4 -> 16.4 us with 64 buckets).
// Alone, the plan keeps one bucket per SM, its fastest grid.
constexpr int kBesideLookupBuckets = 64;

cudaError_t launch_embed_fwd_plan(const vce_problem& p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                                  int32_t* local, void* ws, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  if (cudaError_t e = plan_multi(&p, &ids, &ws, 1, kBesideLookupBuckets, st)) return e;
  const int esize = p.dtype == VCE_BF16 ? 2 : 4;
  const int row_vecs = static_cast<int>(p.H * esize / 16);
  const int64_t blocks = ceil_div(p.T, kGatherWarps);
  const cudaError_t e = launch_dependent(embed_gather_kernel<true>, dim3(static_cast<unsigned>(blocks)),
                                         dim3(kGatherWarps * 32), 0, st, ids, static_cast<const uint4*>(W),
                                         static_cast<uint4*>(E), owner, local, p.T, p.Vp, p.V_real, p.S, row_vecs);
  note_launch(VCE_K_EMBED_GATHER, st);
  return e;
}

size_t embed_bwd_ws_bytes(const vce_problem& p) { return bwd_layout(p).total; }

bool embed_bwd_supported(const vce_problem& p) {   // the reduce numbers its items (<= T * nhm) in 32 bits
  return static_cast<int64_t>(p.T) * bwd_layout(p).nhm < (int64_t(1) << 31);
}

namespace {

EmbSlot emb_slot(const vce_problem& p, void* ws, float* dW) {
  const BwdLayout L = bwd_layout(p);
  char* b = static_cast<char*>(ws);
  EmbSlot sl;
  sl.hdr = reinterpret_cast<int32_t*>(b + L.hdr);
  sl.rows = static_cast<int32_t>(p.V_real);
  sl.tsorted = reinterpret_cast<const int32_t*>(b + L.tsorted);
  sl.runs = reinterpret_cast<const RunDesc*>(b + L.runs);
  sl.dW = dW;
  sl.partials = reinterpret_cast<float*>(b + L.partials);
  sl.counters = reinterpret_cast<int32_t*>(b + L.counters);
  return sl;
}

enum class SortPath { kCount, kBucket, kSmem, kGlobal };

SortPath sort_path(const vce_problem& p, int nb, int cl) {
  const int tbits = bit_width(p.T);
  const int qbits = bit_width(ceil_div(p.V_real, nb));
  // The bucketed sorts divide ids by NB with a multiply-high, exact for ids
  // below 2^32 / NB; keys (q << tbits) | t stay below the all-ones word that
  // marks "not mine".
  const bool magic_ok = static_cast<uint64_t>(p.V_real) * static_cast<uint64_t>(nb) <= (uint64_t(1) << 32);
  const bool bucketed = p.T <= kSmemSortMax && tbits + qbits <= 31 && nb > 1 && magic_ok;
  if (bucketed) return count_sort_smem(p.T, ceil_div(p.V_real, nb), cl) <= kCountSmemBudget ? SortPath::kCount
                                                                                           : SortPath::kBucket;
  if (p.T <= kSmemSortMax && tbits + bit_width(p.V_real) <= 32) return SortPath::kSmem;
  return SortPath::kGlobal;
}

// The counting sort's choice for one problem: its path, its bucket count NB
// (the grid) and its cluster size.
struct SortPlan {
  SortPath path;
  int nb, cl;
};

constexpr int kSortCluster = 8;
constexpr int kClusterRounds = (kSmemSortMax / kSortCluster + 1023) / 1024;   // rounds per warp at most

using CountKern = void (*)(const SortJobs, int, int, int, uint32_t);

void set_count_smem_limit(CountKern k, cudaError_t* err) {
  const cudaError_t e =
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kCountSmemBudget));
  if (e != cudaSuccess && *err == cudaSuccess) *err = e;
}

// Buckets of the clustered counting sort on the current device: kSortCluster
// times the clusters of one-CTA-per-SM sort blocks that can be resident at
// once (0 if none can), so that the grid runs in one wave.
int cluster_sort_buckets(cudaError_t* err) {
  static std::atomic<uint64_t> configured{0};
  static std::atomic<int> buckets[64];   // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 0;
  if (device_pending(configured)) {
    for (auto k : {embed_sort_count_kernel<2, 1>, embed_sort_count_kernel<4, 1>, embed_sort_count_kernel<8, 1>,
                   embed_sort_count_kernel<16, 1>, embed_sort_count_kernel<1, kSortCluster>,
                   embed_sort_count_kernel<2, kSortCluster>, embed_sort_count_kernel<kClusterRounds, kSortCluster>})
      set_count_smem_limit(k, err);
    if (*err != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSortCluster * 64);
    cfg.blockDim = dim3(kBktThreads);
    cfg.dynamicSmemBytes = kCountSmemBudget;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSortCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, embed_sort_count_kernel<2, kSortCluster>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();   // no clusters of this size: the one-CTA load stays
      n = 0;
    }
    buckets[dev].store(n * kSortCluster);
    mark_device_done(configured);
  }
  return buckets[dev].load();
}

// The clustered load pays off once every CTA would load more than 8192 ids
// (16 rounds per warp): measured on GB300, about 3 us less for 16384 tokens
// and about 1 us more for 8192. VCE_EMBED_SORT_CLUSTER=1 in the environment
// takes it whenever the counting sort runs, =0 never.
SortPlan plan_sort(const vce_problem& p, int num_sms, int max_nb, cudaError_t* err) {
  const char* env = std::getenv("VCE_EMBED_SORT_CLUSTER");
  const bool set = env && (env[0] == '0' || env[0] == '1') && env[1] == 0;
  const bool allow = set ? env[0] == '1' : p.T > 8192;
  const int nbc = cluster_sort_buckets(err);
  if (allow && nbc >= 2 * kSortCluster && sort_path(p, nbc, kSortCluster) == SortPath::kCount)
    return {SortPath::kCount, nbc, kSortCluster};
  int nb = num_sms > 0 ? num_sms : 1;
  if (max_nb > 0 && nb > max_nb) nb = max_nb;
  return {sort_path(p, nb, 1), nb, 1};
}

// The column slices of multi-run ids' items. Narrow ones (half a wide slice)
// when one problem's dE is at most 64 MB: there the call's time is set by the
// hottest id's chain of dependent loads (its run's rows, then its run sums),
// which narrow items halve; on larger problems the call is bound by HBM and
// the extra items cost more than the shorter chain saves (measured on GB300:
// 8192 x 2048 tokens x columns 26.6 -> 22.5 us, 16384 x 3072 38.9 -> 41.0 us).
// VCE_EMBED_NARROW=1 or =0 in the environment forces or forbids them. The
// plan and its application must agree: the plan records the slice count.
struct FrontSlices {
  int nhf;
  bool narrow;
};
constexpr int64_t kNarrowMaxBytes = int64_t(64) << 20;
FrontSlices front_slices(const vce_problem& p, int n_problems) {
  const BwdLayout L = bwd_layout(p);
  const char* env = std::getenv("VCE_EMBED_NARROW");
  const bool set = env && (env[0] == '0' || env[0] == '1') && env[1] == 0;
  const int64_t esize = p.dtype == VCE_BF16 ? 2 : 4;
  const bool narrow = set ? env[0] == '1' : (n_problems == 1 && p.T * p.H * esize <= kNarrowMaxBytes);
  return narrow ? FrontSlices{L.nhm, true} : FrontSlices{L.nh, false};
}

// One launch of the counting sort over n problems of the same T (ps, their
// ids and workspaces), nb buckets each, in clusters of cl CTAs (nb a multiple
// of cl), with counters for nhf column slices per multi-run id.
cudaError_t launch_count_sort(const vce_problem* ps, const int64_t* const* ids, void* const* ws, int n, int nb, int cl,
                              int nhf, cudaStream_t st) {
  if (n < 1 || n > kMaxSortJobs || nb < 2 || nb % cl != 0) return cudaErrorInvalidValue;
  const int64_t T = ps[0].T;
  SortJobs J{};
  J.nb = nb;
  size_t smem = 0;
  for (int k = 0; k < n; ++k) {
    const BwdLayout L = bwd_layout(ps[k]);
    char* b = static_cast<char*>(ws[k]);
    J.ids[k] = ids[k];
    J.V_real[k] = ps[k].V_real;
    J.nq[k] = static_cast<int>(ceil_div(ps[k].V_real, nb));
    J.hdr[k] = reinterpret_cast<int32_t*>(b + L.hdr);
    J.tsorted[k] = reinterpret_cast<int32_t*>(b + L.tsorted);
    J.runs[k] = reinterpret_cast<RunDesc*>(b + L.runs);
    J.counters[k] = reinterpret_cast<int32_t*>(b + L.counters);
    const size_t sm = count_sort_smem(T, J.nq[k], cl);
    if (sm > smem) smem = sm;
  }
  const uint32_t nb_magic = 0xFFFFFFFFu / static_cast<uint32_t>(nb) + 1u;   // floor((2^32 - 1) / NB) + 1
  CountKern kern;
  if (cl == 1) {
    // Phase A's rounds of 32 tokens per warp: 2, 4, 8 or 16.
    const int rounds = T <= 2048 ? 2 : T <= 4096 ? 4 : T <= 8192 ? 8 : 16;
    kern = rounds == 2   ? embed_sort_count_kernel<2, 1>
           : rounds == 4 ? embed_sort_count_kernel<4, 1>
           : rounds == 8 ? embed_sort_count_kernel<8, 1>
                         : embed_sort_count_kernel<16, 1>;
  } else {
    // Each rank loads a segment of Tc <= 16384 / kSortCluster tokens: up to 512 / kSortCluster rounds per warp.
    const int tc = count_seg_cap(static_cast<int>(T), kSortCluster);
    const int tpw = ((tc + kBktWarps - 1) / kBktWarps + 31) & ~31;
    if (cl != kSortCluster || tpw > 32 * kClusterRounds) return cudaErrorInvalidValue;
    kern = tpw <= 32 ? embed_sort_count_kernel<1, kSortCluster>
           : tpw <= 64 ? embed_sort_count_kernel<2, kSortCluster>
                       : embed_sort_count_kernel<kClusterRounds, kSortCluster>;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n * nb));
  cfg.blockDim = dim3(kBktThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cl > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, J, static_cast<int>(T), bit_width(T), nhf, nb_magic);
}

// Sorts one problem's valid (id, t) pairs into its workspace and builds its
// runs, with counters for nhf column slices per multi-run id. A bucketed sort
// needs its header zeroed by the kernel before it.
cudaError_t launch_sort(const vce_problem& p, const int64_t* ids, void* ws, const SortPlan& plan, int nhf,
                        cudaStream_t st) {
  const SortPath path = plan.path;
  const int nb = plan.nb;
  const BwdLayout L = bwd_layout(p);
  char* b = static_cast<char*>(ws);
  int32_t* hdr = reinterpret_cast<int32_t*>(b + L.hdr);
  uint64_t* ka = reinterpret_cast<uint64_t*>(b + L.keys_a);
  uint64_t* kb = reinterpret_cast<uint64_t*>(b + L.keys_b);
  int32_t* seg = reinterpret_cast<int32_t*>(b + L.seg_start);
  int32_t* tsorted = reinterpret_cast<int32_t*>(b + L.tsorted);
  RunDesc* runs = reinterpret_cast<RunDesc*>(b + L.runs);
  int32_t* counters = reinterpret_cast<int32_t*>(b + L.counters);
  const int tbits = bit_width(p.T);
  const int qbits = bit_width(ceil_div(p.V_real, nb));
  const uint32_t nb_magic = 0xFFFFFFFFu / static_cast<uint32_t>(nb > 1 ? nb : 2) + 1u;   // floor((2^32 - 1) / NB) + 1
  if (path == SortPath::kCount) {
    if (cudaError_t e = launch_count_sort(&p, &ids, &ws, 1, nb, plan.cl, nhf, st)) return e;
  } else if (path == SortPath::kBucket) {
    static std::atomic<uint64_t> configured{0};
    if (device_pending(configured)) {
      cudaError_t e = cudaFuncSetAttribute(embed_sort_bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(bucket_sort_smem(kSmemSortMax)));
      if (e != cudaSuccess) return e;
      mark_device_done(configured);
    }
    if (cudaError_t e = launch_dependent(embed_sort_bucket_kernel, dim3(nb), dim3(kBktThreads), bucket_sort_smem(p.T),
                                         st, ids, static_cast<int>(p.T), p.V_real, tbits, qbits, nhf, nb_magic, hdr,
                                         tsorted, runs, counters))
      return e;
  } else if (path == SortPath::kSmem) {
    static std::atomic<uint64_t> configured{0};
    if (device_pending(configured)) {
      cudaError_t e = cudaFuncSetAttribute(embed_sort_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemSortBytes));
      if (e != cudaSuccess) return e;
      mark_device_done(configured);
    }
    embed_sort_smem_kernel<<<1, kSortThreads, kSmemSortBytes, st>>>(ids, static_cast<int>(p.T), p.V_real, tbits,
                                                                    bit_width(p.V_real), nhf, hdr, tsorted, runs,
                                                                    counters);
  } else {
    embed_sort_kernel<<<1, kSortThreads, 0, st>>>(ids, p.T, p.V_real, nhf, hdr, ka, kb, seg, tsorted, runs,
                                                  counters);
  }
  note_launch(path == SortPath::kCount && plan.cl > 1 ? VCE_K_EMBED_SORT_CLUSTER : VCE_K_EMBED_SORT, st);
  return cudaGetLastError();
}

// One reduce over the sorted problems in `sl` (all with p's T, H and dtype).
cudaError_t launch_reduce(const vce_problem& p, const EmbSlots& sl, const void* dE, int32_t* status,
                          cudaStream_t st) {
  const BwdLayout L = bwd_layout(p);
  const DevInfo di = current_device_info();
  const int grid = di.num_sms * 8;
  // Items of one problem number at most T * nhm (a run per token at most); the
  // multiply-high gives item / d exactly for items below 2^32 / d.
  const uint64_t max_items = static_cast<uint64_t>(p.T) * static_cast<uint64_t>(L.nhm);
  auto magic = [&](int d) -> uint32_t {
    return (d > 1 && max_items * static_cast<uint64_t>(d) < (uint64_t(1) << 32))
               ? 0xFFFFFFFFu / static_cast<uint32_t>(d) + 1u
               : 0u;
  };
  const FrontSlices fs = front_slices(p, sl.n);
  const uint32_t nh_magic = magic(L.nh), nhf_magic = magic(fs.nhf);
  // One problem reads dE once; the n-gram tables read it once each.
  const bool stream = sl.n == 1;
  const int H = static_cast<int>(p.H), cap = static_cast<int>(p.T);
  cudaError_t e;
  if (p.dtype == VCE_BF16) {
    const uint16_t* d = static_cast<const uint16_t*>(dE);
    if (fs.narrow)
      e = launch_dependent(
          stream ? embed_reduce_narrow_kernel<uint16_t, true> : embed_reduce_narrow_kernel<uint16_t, false>,
          dim3(grid), dim3(128), 0, st, sl, d, H, L.nh, nh_magic, fs.nhf, nhf_magic, cap, status);
    else
      e = launch_dependent(stream ? embed_reduce_kernel<uint16_t, true> : embed_reduce_kernel<uint16_t, false>,
                           dim3(grid), dim3(128), 0, st, sl, d, H, L.nh, nh_magic, cap, status);
  } else {
    const float* d = static_cast<const float*>(dE);
    if (fs.narrow)
      e = launch_dependent(stream ? embed_reduce_narrow_kernel<float, true> : embed_reduce_narrow_kernel<float, false>,
                           dim3(grid), dim3(128), 0, st, sl, d, H, L.nh, nh_magic, fs.nhf, nhf_magic, cap, status);
    else
      e = launch_dependent(stream ? embed_reduce_kernel<float, true> : embed_reduce_kernel<float, false>, dim3(grid),
                           dim3(128), 0, st, sl, d, H, L.nh, nh_magic, cap, status);
  }
  note_launch(VCE_K_EMBED_REDUCE, st);
  return e;
}

}  // namespace

namespace {

// The plans of n problems: one header-zeroing launch (for the bucketed
// sorts), then the sorts (side by side in one launch where they allow it,
// below; else one per problem), a one-CTA-per-bucket grid capped at
// max_nb buckets when it runs without clusters (0: one bucket per SM). Any
// bucket count gives the same plan up to the order of the runs in the list,
// and the same results.
cudaError_t plan_multi(const vce_problem* ps, const int64_t* const* ids, void* const* ws, int n, int max_nb,
                       cudaStream_t st) {
  if (n < 1 || n > kMaxSlots) return cudaErrorInvalidValue;
  if (ps[0].T == 0) return cudaSuccess;
  const DevInfo di = current_device_info();
  SortPlan plan[kMaxSlots];
  int32_t* zero[kMaxSlots] = {nullptr, nullptr, nullptr};
  bool any_bucketed = false;
  for (int k = 0; k < n; ++k) {
    cudaError_t err = cudaSuccess;
    plan[k] = plan_sort(ps[k], di.num_sms, max_nb, &err);
    if (err != cudaSuccess) return err;
    if (plan[k].path == SortPath::kCount || plan[k].path == SortPath::kBucket) {
      zero[k] = emb_slot(ps[k], ws[k], nullptr).hdr;
      any_bucketed = true;
    }
  }
  if (any_bucketed) {
    embed_hdr_zero_kernel<<<1, 64, 0, st>>>(zero[0], zero[1], zero[2]);
    note_launch(VCE_K_EMBED_HDR, st);
    if (cudaError_t e = cudaGetLastError()) return e;
  }
  // Problems of the same T whose sorts all take the counting path with the
  // same cluster size (the n-gram tables) are sorted side by side by one
  // launch, the buckets shared out among them: each sort CTA loads every id
  // whatever its bucket count, so fewer buckets per problem cost little, while
  // one sort after another would each take every SM for the length of a sort.
  if (n > 1) {
    bool joint = true;
    for (int k = 0; k < n; ++k)
      joint = joint && plan[k].path == SortPath::kCount && plan[k].cl == plan[0].cl && ps[k].T == ps[0].T;
    const int cl = plan[0].cl;
    const int nbj = ((plan[0].nb / cl) / n) * cl;
    for (int k = 0; joint && k < n; ++k) joint = nbj >= 2 && sort_path(ps[k], nbj, cl) == SortPath::kCount;
    if (joint) return launch_count_sort(ps, ids, ws, n, nbj, cl, front_slices(ps[0], n).nhf, st);
  }
  for (int k = 0; k < n; ++k)
    if (cudaError_t e = launch_sort(ps[k], ids[k], ws[k], plan[k], front_slices(ps[k], n).nhf, st)) return e;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_embed_bwd_plan_multi(const vce_problem* ps, const int64_t* const* ids, void* const* ws, int n,
                                        cudaStream_t st) {
  return plan_multi(ps, ids, ws, n, 0, st);
}

cudaError_t launch_embed_bwd_apply_multi(const vce_problem* ps, float* const* dW, void* const* ws, int n,
                                         const void* dE, int32_t* status, cudaStream_t st) {
  if (n < 1 || n > kMaxSlots) return cudaErrorInvalidValue;
  if (ps[0].T == 0) return cudaSuccess;
  EmbSlots sl{};
  sl.n = n;
  for (int k = 0; k < n; ++k) sl.s[k] = emb_slot(ps[k], ws[k], dW[k]);
  return launch_reduce(ps[0], sl, dE, status, st);
}

cudaError_t launch_embed_bwd_multi(const vce_problem* ps, const int64_t* const* ids, float* const* dW,
                                   void* const* ws, int n, const void* dE, int32_t* status, cudaStream_t st) {
  if (cudaError_t e = launch_embed_bwd_plan_multi(ps, ids, ws, n, st)) return e;
  return launch_embed_bwd_apply_multi(ps, dW, ws, n, dE, status, st);
}

cudaError_t launch_embed_bwd(const vce_problem& p, const int64_t* ids, const void* dE, float* dW, void* ws,
                             int32_t* status, cudaStream_t st) {
  return launch_embed_bwd_multi(&p, &ids, &dW, &ws, 1, dE, status, st);
}

cudaError_t launch_embed_bwd_plan(const vce_problem& p, const int64_t* ids, void* ws, cudaStream_t st) {
  return launch_embed_bwd_plan_multi(&p, &ids, &ws, 1, st);
}

cudaError_t launch_embed_bwd_apply(const vce_problem& p, const void* dE, float* dW, void* ws, int32_t* status,
                                   cudaStream_t st) {
  return launch_embed_bwd_apply_multi(&p, &dW, &ws, 1, dE, status, st);
}

}  // namespace vce
