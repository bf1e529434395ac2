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
// owned row): the valid (id, t) pairs are sorted (stable LSD radix sort on the
// id, one CTA), the tokens of each id are cut into runs of kEmbedBwdChunk,
// each run is summed in fp32 in ascending t, run sums are combined left to
// right, and the total is added once into the fp32 row. The order is fixed,
// so results are bit-identical from run to run.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace vce {
namespace {

// ---------------------------------------------------------------------------
// Forward gather: one warp per token row.
// ---------------------------------------------------------------------------
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32)
    embed_gather_kernel(const int64_t* __restrict__ ids, const uint4* __restrict__ W, uint4* __restrict__ E,
                        int32_t* __restrict__ owner, int32_t* __restrict__ local, int64_t T, int64_t Vp,
                        int64_t V_real, int32_t S, int row_vecs) {
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
constexpr int kSmemItems = kSmemSortMax / kSortThreads;   // 16 keys per thread
// Shared-memory arrays are padded by one word per 32 (index i at i + i/32), so
// that each thread's 16 consecutive entries fall in distinct banks across a warp.
__host__ __device__ constexpr int pad32(int i) { return i + (i >> 5); }
constexpr size_t kSmemSortBytes = 2 * pad32(kSmemSortMax) * sizeof(uint32_t) +
                                  pad32(16 * kSortThreads) * sizeof(int) + 64 * sizeof(int);

struct RunDesc {
  int32_t start, end;   // sorted positions [start, end)
  int32_t id;
  int32_t slot;         // partial slot (multi-run ids) or -1
  int32_t mseg;         // index of the multi-run id, or -1
  int32_t nruns;        // runs of this id
  int32_t first_slot;   // slot of the id's first run
  int32_t pad;
};

struct BwdLayout {
  size_t hdr, keys_a, keys_b, seg_start, tsorted, runs, counters, partials, total;
  int64_t n_counters, n_slots;
  int nh;
};

int cols_per_item(int esize) { return 128 * (16 / esize); }

BwdLayout bwd_layout(const vce_problem& p) {
  BwdLayout L{};
  const int64_t T = p.T;
  const int esize = p.dtype == VCE_BF16 ? 2 : 4;
  L.nh = static_cast<int>(ceil_div(p.H, cols_per_item(esize)));
  L.n_counters = (T / (kEmbedBwdChunk + 1) + 2) * L.nh;
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

// Block-wide exclusive scan of one int per thread (1024 threads).
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
    int w = sh_warp[lane];
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

// Runs of kEmbedBwdChunk tokens for the segments [s0, s0 + per_thread) of one
// thread (all threads together cover [0, nseg) in order); slots for multi-run
// ids. seg[s] is the sorted position where segment s starts (segment s ends at
// seg[s + 1], the last one at n); id_of(s) gives its id.
template <typename SegAt, typename IdOf>
__device__ __forceinline__ void build_runs(SegAt seg, int nseg, int n, int per_thread, int nh, IdOf id_of,
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
  int r0 = block_excl_scan(my_runs, sh_warp, &t_runs);
  int m0 = block_excl_scan(my_multi, sh_warp, &t_multi);
  int q0 = block_excl_scan(my_slots, sh_warp, &t_slots);
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
      runs[r0 + k] = r;
    }
    if (multi) {
      for (int hh = 0; hh < nh; ++hh) counters[m0 * nh + hh] = 0;
      m0 += 1;
      q0 += nr;
    }
    r0 += nr;
  }
  if (threadIdx.x == 0) {
    hdr[1] = t_runs;
    hdr[3] = t_multi;
    hdr[4] = t_slots;
  }
}

// Shared-memory variant: keys (id << tbits) | t in 32 bits, T <= kSmemSortMax.
__global__ void __launch_bounds__(kSortThreads, 1)
    embed_sort_smem_kernel(const int64_t* __restrict__ ids, int T, int64_t V_real, int tbits, int idbits, int nh,
                           int32_t* hdr, int32_t* tsorted, RunDesc* runs, int32_t* counters) {
  extern __shared__ __align__(16) uint32_t smem_keys[];
  uint32_t* ka = smem_keys;
  uint32_t* kb = smem_keys + pad32(kSmemSortMax);
  int* ctab = reinterpret_cast<int*>(smem_keys + 2 * pad32(kSmemSortMax));   // [16 digits][1024 threads]
  int* sh_warp = ctab + pad32(16 * kSortThreads);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;

  // Phase 0: stable compaction of the valid ids. Warp w reads its contiguous
  // block of tokens 32 at a time (coalesced); ballots give the order.
  const int tpw = ((T + kSortWarps - 1) / kSortWarps + 31) / 32 * 32;   // tokens per warp, <= 512
  int wcount = 0;
  for (int j = 0; j < tpw / 32; ++j) {
    const int t = warp * tpw + j * 32 + lane;
    const int64_t id = t < T ? ids[t] : -1;
    wcount += __popc(__ballot_sync(0xffffffffu, id >= 0 && id < V_real));
  }
  if (lane == 0) sh_warp[warp] = wcount;
  __syncthreads();
  int wbase = 0, n = 0;
  for (int w = 0; w < kSortWarps; ++w) {
    const int c = sh_warp[w];
    wbase += w < warp ? c : 0;
    n += c;
  }
  __syncthreads();
  for (int j = 0; j < tpw / 32; ++j) {
    const int t = warp * tpw + j * 32 + lane;
    const int64_t id = t < T ? ids[t] : -1;
    const bool ok = id >= 0 && id < V_real;
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (ok) ka[pad32(wbase + __popc(bal & lt_mask))] = (static_cast<uint32_t>(id) << tbits) | static_cast<uint32_t>(t);
    wbase += __popc(bal);
  }
  __syncthreads();

  // Phase 1: stable LSD radix passes over the id bits, 4 bits per pass. Thread
  // tid owns kpt consecutive keys and ranks them with its own shared-memory
  // counter per digit; the table of counters (digit-major, thread-minor) is
  // scanned once per pass, which gives every key its stable destination.
  const int kpt = (n + kSortThreads - 1) / kSortThreads;   // keys per thread, <= 16
  const int k0 = tid * kpt;
  uint32_t* src = ka;
  uint32_t* dst = kb;
  for (int shift = tbits; shift < tbits + idbits; shift += 4) {
    uint32_t key[kSmemItems];
    uint32_t lrw[kSmemItems / 4] = {};   // byte j%4 of word j/4: rank among this thread's keys of that digit
#pragma unroll
    for (int b = 0; b < 16; ++b) ctab[pad32(b * kSortThreads + tid)] = 0;
#pragma unroll
    for (int j = 0; j < kSmemItems; ++j) {
      const bool ok = j < kpt && k0 + j < n;
      key[j] = ok ? src[pad32(k0 + j)] : 0u;
      if (ok) {
        int* c = &ctab[pad32(static_cast<int>((key[j] >> shift) & 15u) * kSortThreads + tid)];
        const int v = *c;
        *c = v + 1;
        lrw[j >> 2] |= static_cast<uint32_t>(v) << ((j & 3) * 8);
      }
    }
    __syncthreads();
    {
      int v[16];
      int sum = 0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        v[k] = ctab[pad32(tid * 16 + k)];
        sum += v[k];
      }
      int all;
      int run = block_excl_scan(sum, sh_warp, &all);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        ctab[pad32(tid * 16 + k)] = run;
        run += v[k];
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kSmemItems; ++j)
      if (j < kpt && k0 + j < n)
        dst[pad32(ctab[pad32(static_cast<int>((key[j] >> shift) & 15u) * kSortThreads + tid)] +
                  static_cast<int>((lrw[j >> 2] >> ((j & 3) * 8)) & 0xFFu))] = key[j];
    __syncthreads();
    uint32_t* tmp = src;
    src = dst;
    dst = tmp;
  }

  // Phase 2: sorted token indices to global memory; segment starts into the
  // free key buffer (seg), one entry per distinct id, at most n <= 16384.
  const uint32_t tmask = (1u << tbits) - 1u;
  int* seg = reinterpret_cast<int*>(dst);
  int heads = 0;
  for (int j = 0; j < kpt; ++j) {
    const int q = k0 + j;
    if (q < n) {
      tsorted[q] = static_cast<int32_t>(src[pad32(q)] & tmask);
      if (q == 0 || (src[pad32(q)] >> tbits) != (src[pad32(q - 1)] >> tbits)) ++heads;
    }
  }
  int nseg;
  int sidx = block_excl_scan(heads, sh_warp, &nseg);
  for (int j = 0; j < kpt; ++j) {
    const int q = k0 + j;
    if (q < n && (q == 0 || (src[pad32(q)] >> tbits) != (src[pad32(q - 1)] >> tbits))) seg[pad32(sidx++)] = q;
  }
  __syncthreads();

  // Phase 3: runs of kEmbedBwdChunk tokens. Per segment s: nr runs; packed
  // prefix rb[s] = (runs before s) << 16 | (multi-run segments before s) in
  // ctab. Then each run is written by one thread, which finds its segment by
  // binary search.
  auto seg_end = [&](int sg) { return sg + 1 < nseg ? seg[pad32(sg + 1)] : n; };
  const int spt = (nseg + kSortThreads - 1) / kSortThreads;   // segments per thread, <= 16
  const int s0 = tid * spt;
  int packed = 0;
  for (int j = 0; j < spt; ++j) {
    const int sg = s0 + j;
    if (sg < nseg) {
      const int nr = (seg_end(sg) - seg[pad32(sg)] + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
      packed += (nr << 16) | (nr > 1 ? 1 : 0);
    }
  }
  int tot_packed;
  int pre = block_excl_scan(packed, sh_warp, &tot_packed);
  for (int j = 0; j < spt; ++j) {
    const int sg = s0 + j;
    if (sg < nseg) {
      ctab[pad32(sg)] = pre;
      const int nr = (seg_end(sg) - seg[pad32(sg)] + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
      pre += (nr << 16) | (nr > 1 ? 1 : 0);
    }
  }
  __syncthreads();
  const int n_runs = tot_packed >> 16, n_multi = tot_packed & 0xFFFF;
  for (int r = tid; r < n_runs; r += kSortThreads) {
    int lo = 0, hi = nseg - 1;   // largest sg with runs-before(sg) <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((ctab[pad32(mid)] >> 16) <= r)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int sg = lo;
    const int rb = ctab[pad32(sg)] >> 16, mb = ctab[pad32(sg)] & 0xFFFF;
    const int st = seg[pad32(sg)], en = seg_end(sg);
    const int nr = (en - st + kEmbedBwdChunk - 1) / kEmbedBwdChunk;
    const int k = r - rb;
    const bool multi = nr > 1;
    const int q0 = rb - (sg - mb);   // slots used by the multi-run segments before sg
    RunDesc rd;
    rd.start = st + k * kEmbedBwdChunk;
    rd.end = min(en, rd.start + kEmbedBwdChunk);
    rd.id = static_cast<int32_t>(src[pad32(st)] >> tbits);
    rd.slot = multi ? q0 + k : -1;
    rd.mseg = multi ? mb : -1;
    rd.nruns = nr;
    rd.first_slot = multi ? q0 : -1;
    rd.pad = 0;
    runs[r] = rd;
    if (multi && k == 0)
      for (int hh = 0; hh < nh; ++hh) counters[mb * nh + hh] = 0;
  }
  if (tid == 0) {
    hdr[0] = n;
    hdr[1] = n_runs;
    hdr[2] = nseg;
    hdr[3] = n_multi;
    hdr[4] = (tot_packed >> 16) - (nseg - n_multi);
  }
}

// Workspace variant: 64-bit keys (id << 32) | t, any T.
__global__ void __launch_bounds__(kSortThreads, 1)
    embed_sort_kernel(const int64_t* __restrict__ ids, int64_t T, int64_t V_real, int nh, int32_t* hdr,
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
  build_runs(seg_at, nseg, n, (nseg + kSortThreads - 1) / kSortThreads, nh, id_of, sh_warp, hdr, runs,
             counters);
  if (tid == 0) {
    hdr[0] = n;
    hdr[2] = nseg;
  }
}

// ---------------------------------------------------------------------------
// Backward, step 2: persistent segmented reduction. Work item = (run, column
// slice of 128 threads x 16 bytes).
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

template <typename TE>
__global__ void __launch_bounds__(128)
    embed_reduce_kernel(const int32_t* __restrict__ hdr, const int32_t* __restrict__ tsorted,
                        const RunDesc* __restrict__ runs, const TE* __restrict__ dE, float* __restrict__ dW,
                        float* partials, int32_t* counters, int H, int nh) {
  constexpr int VEC = 16 / sizeof(TE);
  constexpr int NQ = VEC / 4;
  constexpr int U = 8;   // rows loaded ahead of the sequential adds
  __shared__ int s_last;
  const int lane = threadIdx.x & 31;
  const int n_items = hdr[1] * nh;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int r = item / nh, hs = item - r * nh;
    const RunDesc rd = runs[r];
    const int len = rd.end - rd.start;   // <= 32
    const int col = hs * 128 * VEC + static_cast<int>(threadIdx.x) * VEC;
    const bool active = col < H;
    // the run's token indices, one per lane, broadcast below
    const int my_t = lane < len ? tsorted[rd.start + lane] : 0;
    float4* row = reinterpret_cast<float4*>(dW + static_cast<int64_t>(rd.id) * H + col);
    float4 w[NQ];
    if (rd.slot < 0 && active) {   // single-run id: fetch the row now, add once the sum is ready
#pragma unroll
      for (int q = 0; q < NQ; ++q) w[q] = row[q];
    }
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
    for (int p = 0; p < len; p += U) {
      uint4 v[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int t = __shfl_sync(0xffffffffu, my_t, (p + k) & 31);
        v[k] = make_uint4(0, 0, 0, 0);
        if (active && p + k < len) v[k] = __ldg(reinterpret_cast<const uint4*>(dE + static_cast<int64_t>(t) * H + col));
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (p + k < len) {          // tokens in ascending t, one add each
          float f[VEC];
          widen<TE>(v[k], f);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] = acc[e] + f[e];
        }
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
        for (int j = 1; j < rd.nruns; ++j) {
          const float4* sj =
              reinterpret_cast<const float4*>(partials + static_cast<int64_t>(rd.first_slot + j) * H + col);
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            float4 a = __ldcg(sj + q);
            tot[4 * q] = tot[4 * q] + a.x;
            tot[4 * q + 1] = tot[4 * q + 1] + a.y;
            tot[4 * q + 2] = tot[4 * q + 2] + a.z;
            tot[4 * q + 3] = tot[4 * q + 3] + a.w;
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
  }
}

}  // namespace

cudaError_t launch_embed_fwd(const vce_problem& p, const int64_t* ids, const void* W, void* E, int32_t* owner,
                             int32_t* local, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  const int esize = p.dtype == VCE_BF16 ? 2 : 4;
  const int row_vecs = static_cast<int>(p.H * esize / 16);
  const int64_t blocks = ceil_div(p.T, kGatherWarps);
  embed_gather_kernel<<<static_cast<unsigned>(blocks), kGatherWarps * 32, 0, st>>>(
      ids, static_cast<const uint4*>(W), static_cast<uint4*>(E), owner, local, p.T, p.Vp, p.V_real, p.S,
      row_vecs);
  note_launch(VCE_K_EMBED_GATHER, st);
  return cudaGetLastError();
}

size_t embed_bwd_ws_bytes(const vce_problem& p) { return bwd_layout(p).total; }

cudaError_t launch_embed_bwd(const vce_problem& p, const int64_t* ids, const void* dE, float* dW, void* ws,
                             int32_t* status, cudaStream_t st) {
  (void)status;
  if (p.T == 0) return cudaSuccess;
  const BwdLayout L = bwd_layout(p);
  char* b = static_cast<char*>(ws);
  int32_t* hdr = reinterpret_cast<int32_t*>(b + L.hdr);
  uint64_t* ka = reinterpret_cast<uint64_t*>(b + L.keys_a);
  uint64_t* kb = reinterpret_cast<uint64_t*>(b + L.keys_b);
  int32_t* seg = reinterpret_cast<int32_t*>(b + L.seg_start);
  int32_t* tsorted = reinterpret_cast<int32_t*>(b + L.tsorted);
  RunDesc* runs = reinterpret_cast<RunDesc*>(b + L.runs);
  int32_t* counters = reinterpret_cast<int32_t*>(b + L.counters);
  float* partials = reinterpret_cast<float*>(b + L.partials);
  const int tbits = bit_width(p.T);
  const int idbits = bit_width(p.V_real);
  if (p.T <= kSmemSortMax && tbits + idbits <= 32) {
    static bool configured = false;
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(embed_sort_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemSortBytes));
      if (e != cudaSuccess) return e;
      configured = true;
    }
    embed_sort_smem_kernel<<<1, kSortThreads, kSmemSortBytes, st>>>(ids, static_cast<int>(p.T), p.V_real, tbits,
                                                                    idbits, L.nh, hdr, tsorted, runs, counters);
  } else {
    embed_sort_kernel<<<1, kSortThreads, 0, st>>>(ids, p.T, p.V_real, L.nh, hdr, ka, kb, seg, tsorted, runs,
                                                  counters);
  }
  note_launch(VCE_K_EMBED_SORT, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const DevInfo di = current_device_info();
  const int grid = di.num_sms * 8;
  if (p.dtype == VCE_BF16)
    embed_reduce_kernel<uint16_t><<<grid, 128, 0, st>>>(hdr, tsorted, runs, static_cast<const uint16_t*>(dE), dW,
                                                        partials, counters, static_cast<int>(p.H), L.nh);
  else
    embed_reduce_kernel<float><<<grid, 128, 0, st>>>(hdr, tsorted, runs, static_cast<const float*>(dE), dW,
                                                     partials, counters, static_cast<int>(p.H), L.nh);
  note_launch(VCE_K_EMBED_REDUCE, st);
  return cudaGetLastError();
}

}  // namespace vce
