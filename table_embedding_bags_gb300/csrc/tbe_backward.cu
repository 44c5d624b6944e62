// tbe_backward.cu -- sparse row-gradient backward of table-batched embedding bags.
//
// [FBT] = the page "FBTriton table-batched embeddings: the backward win is a
// threshold moved from 32 to 256".
//
// What is computed ([FBT] "Why the backward is the hard half"): the table
// gradient is zero except on rows some bag read; row r receives
//   row_grad[r, c] = sum_{i : table_row_base[t_i] + id_i = r} w_i * G[b_i, D_offsets[t_i] + c].
// The batch is inverted by sorting: every lookup gets the key
// table_row_base[t] + id (rows of different tables never collide), equal
// keys form runs, and each run is an independent unit reduced without
// atomics on its output row.  Runs are routed by length ([FBT] "Three tiers,
// routed by run length"): a run shorter than the threshold is reduced by
// one warp; a longer run is cut into chunks whose partial sums meet in a
// workspace and are combined by the last chunk to finish, which learns it
// is last from a counter decremented after a device-scope fence ([FBT]
// "Three tiers, routed by run length", the fused tier).
//
// Kernels, in stream order (no host synchronisation anywhere):
//   0. memset of the counter / look-back region of the workspace
//   1. linearize: bag of every position, key = row base + id (or the
//      sentinel total_rows for an id outside its table), bag sample index,
//      and the digit histograms of every radix pass
//   2. one onesweep pass per 8-bit digit: stable LSD radix sort of
//      (key, position) with per-tile digit ranks and a decoupled look-back
//      over tiles taken in launch order (every wait is bounded)
//   3. run-length segmentation: unique rows and run starts (look-back scan)
//   4. classify: long runs are compacted with one atomic per block; the
//      counts stay on the device ([FBT] "Three tiers, routed by run
//      length", the classification kernel); also the per-table run counts
//   5. reduce: one persistent kernel whose warps take work items from a
//      device counter -- first the long-run chunks, then batches of 32
//      consecutive runs whose short runs the warp reduces itself.
#include <algorithm>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// tile sizes and look-back flags
// ---------------------------------------------------------------------------
constexpr int kLinThreads = 256;
constexpr int kLinOffs = 2048;       // bag offsets staged in shared memory (>= the largest tile)

constexpr int kSortThreads = 256;
constexpr int kSegMaxT = 64;         // segmented sort: most tables
constexpr int kSegBk = 512;          // segmented sort: buckets per pass (digits of up to 9 bits)
constexpr int kSortWarps = kSortThreads / 32;

constexpr int kRleThreads = 256;

constexpr int kClsThreads = 256;
constexpr int kRedThreads = 256;
constexpr int kFanIn = 32;           // children per node of the long-run combine tree

constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagInc = 2u << 30;
constexpr uint32_t kValMask = (1u << 30) - 1;
constexpr int kSpinLimit = 1 << 22;  // polls before a wait gives up (TBE_DEV_TIMEOUT)

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits (bounded) for a published look-back word; on time-out it reports
// TBE_DEV_TIMEOUT and returns an inclusive zero so no later tile waits on it.
// Out of line: waiting is the rare path, and inlined copies would only grow
// the hot code that every block fetches.
__device__ __noinline__ uint32_t wait_flag(const uint32_t* p, int32_t* status) {
  const uint32_t v = poll_word(p, kFlagAgg | kFlagInc, kSpinLimit);
  if (v) return v;
  report(status, TBE_DEV_TIMEOUT);
  return kFlagInc;
}

// Whole-window re-reads before a look-back falls back to waiting word by word.
constexpr int kWindowRetries = 8;

// Mask of the window positions 0..q* (q* = nearest predecessor with an
// inclusive word; all 32 positions when there is none).
__device__ __forceinline__ uint32_t window_upto(uint32_t inc) {
  return inc ? (((inc & (0u - inc)) << 1) - 1u) : 0xffffffffu;
}

// Slow path of one look-back window whose words are not all published: walks
// predecessors hi, hi-1, ... (at most 32), waiting on each, and stops at the
// first inclusive word.  Returns (found << 32) | sum.
__device__ __noinline__ unsigned long long lookback_window_slow(const uint32_t* col, size_t stride, int32_t hi,
                                                                int32_t* status) {
  uint32_t sum = 0;
  for (int q = 0; q < 32 && hi - q >= 0; ++q) {
    uint32_t w = ld_relaxed(col + (size_t)(hi - q) * stride);
    if (!(w & (kFlagAgg | kFlagInc))) w = wait_flag(col + (size_t)(hi - q) * stride, status);
    sum += w & kValMask;
    if (w & kFlagInc) return (1ull << 32) | sum;
  }
  return sum;
}

// Look-back words with one word per tile sit 128 bytes apart: with 32 tiles
// sharing a line, every block's stores and the polls of every later block
// queued on the same few L2 lines (~9 us of waiting per tile, measured).
constexpr int kWordStride = 32;

// Exclusive prefix of tile `tile` computed by a whole block of kRleThreads
// threads: thread i reads the word of predecessor tile-1-i (kRleThreads
// predecessors per round, all requested at once), and the block sums the
// words up to the nearest inclusive one.  Word of tile k: words[k *
// kWordStride].  Every thread must call it; `s_lb` is 2 * warps words of
// shared scratch.  Every wait is bounded (wait_flag).
template <int kThreads>
__device__ __forceinline__ uint32_t lookback_block(const uint32_t* words, int32_t tile, int32_t* status,
                                                   uint32_t* s_lb) {
  constexpr int kWarps = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t excl = 0;
  for (int32_t top = tile - 1; top >= 0; top -= kThreads) {
    const int32_t k = top - tid;
    const uint32_t* wk = words + (size_t)max(k, 0) * kWordStride;
    uint32_t v = k >= 0 ? ld_relaxed(wk) : kFlagInc;
    if (!(v & (kFlagAgg | kFlagInc))) v = wait_flag(wk, status);
    const unsigned inc = __ballot_sync(kFull, (v & kFlagInc) != 0);
    if (lane == 0) s_lb[warp] = inc;
    __syncthreads();
    int stop = kThreads - 1;  // block position of the nearest inclusive word
#pragma unroll
    for (int w = kWarps - 1; w >= 0; --w)
      if (s_lb[w]) stop = w * 32 + __ffs(s_lb[w]) - 1;
    uint32_t x = tid <= stop ? (v & kValMask) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    if (lane == 0) s_lb[kWarps + warp] = x;
    __syncthreads();
    uint32_t sum = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sum += s_lb[kWarps + w];
    excl += sum;
    const bool found = stop < kThreads - 1 || s_lb[kWarps - 1] != 0;
    __syncthreads();  // s_lb is reused by the next round
    if (found) break;
  }
  return excl;
}

// Kernels launched with programmatic stream serialisation start while their
// predecessor drains; this waits until the predecessor grid has completed and
// its writes are visible (a no-op for a kernel launched without the attribute).
__device__ __forceinline__ void wait_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream be scheduled once every block of this
// one has started: its blocks then wait in wait_predecessor() for this grid
// to finish instead of being launched after it, which hides the launch gap.
// Correctness does not depend on it (the wait covers completion and memory).
__device__ __forceinline__ void release_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int32_t table_of_row(const TableMeta* meta, int32_t T, int64_t row) {
  int lo = 0, hi = T - 1;  // largest t with row_base[t] <= row
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(&meta[mid].row_base) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct Layout {
  size_t keys_a, keys_b, vals_a, vals_b, bag_of, bag_sorted, psw_sorted, coef, run_starts, run_table, long_list, sub_list,
      gofs, partials;
  size_t zero_begin, hist, sort_tiles, rle_tile, counters, zero_end;
  size_t lin_zero_begin, sort_lookback, rle_lookback, combine, lin_zero_end;
  size_t total;
  int npass, sort_ntiles, rle_ntiles, lin_blocks;
  bool small;  // few tiles per SM: the kernels use half-size tiles
  int seg_dbits;  // > 0: segmented sort in two passes of this many bits
  size_t seg_hist, seg_inv;
  int64_t long_cap, chunk_cap, sub_cap;
  int32_t slot_floats, item_lookups, chunk;
};

// counters: 8-byte slots; kCntLong holds (long runs << 32) | chunks
enum Counter { kCntU = 0, kCntInvalid = 1, kCntWork = 2, kCntSub = 3, kCntLong = 4, kNumCounters = 8 };
// counter k lives at counters[k * kCntStride] (uint32 units): each on its own
// 128-byte line, so the reducer's claims do not slow reads of the others
constexpr int kCntStride = 32;

static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Lookups per long-run chunk: the tuning value, or with 0 a size that keeps
// a few work items per warp of the reduction (64 for small batches, up to
// 256 for large ones, where fewer chunks mean less combining).
static int32_t effective_chunk(const Tuning& tu, int64_t N) {
  if (tu.long_chunk > 0) return tu.long_chunk;
  const int64_t per = N / (4 * 32 * (int64_t)sm_count());
  return (int32_t)std::min<int64_t>(256, std::max<int64_t>(64, per / 32 * 32));
}

Layout make_layout(const Plan& p, int32_t B, int64_t N) {
  (void)B;
  Layout L{};
  const Tuning& tu = tuning();
  L.npass = (p.key_bits + 7) / 8;
  // few tables whose ids need at most 18 bits: two passes over ids within
  // each table replace the passes over global rows
  L.seg_dbits = (p.T < kSegMaxT && p.seg_bits <= 18 && L.npass > 2) ? (p.seg_bits + 1) / 2 : 0;
  // a batch that gives the big tiles fewer than two per SM uses half-size
  // tiles, so more SMs (and more warps per SM) take part
  L.small = N < (int64_t)2 * sm_count() * kSortThreads * 12;
  const int sort_tile = kSortThreads * (L.small ? 6 : 12);
  const int lin_tile = kLinThreads * (L.small ? 4 : 8);
  const int rle_tile = kRleThreads * (L.small ? 4 : 8);
  L.sort_ntiles = (int)((N + sort_tile - 1) / sort_tile);
  if (L.seg_dbits > 0) {  // tiles never span tables: at most one partial tile per table more
    L.npass = 2;
    L.sort_ntiles += p.T;
  }
  L.rle_ntiles = (int)((N + rle_tile - 1) / rle_tile);
  L.lin_blocks = (int)((N + lin_tile - 1) / lin_tile);
  const int64_t tau = std::max(1, tu.long_run_threshold);
  L.chunk = effective_chunk(tu, N);
  const int64_t C = L.chunk;
  L.long_cap = N / tau + 1;
  L.chunk_cap = N / C + L.long_cap + 1;
  // a part holds at least item_lookups lookups except the last of a batch
  L.item_lookups = (int32_t)std::max<int64_t>(tu.short_item_lookups, tau);
  L.sub_cap = (N + 31) / 32 + N / L.item_lookups + 1;
  L.slot_floats = (p.maxD + 3) / 4 * 4;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off += up256(bytes); return o; };
  L.keys_a = take(4 * (size_t)N);
  L.keys_b = take(4 * (size_t)N);
  L.vals_a = take(4 * (size_t)N);
  L.vals_b = take(4 * (size_t)N);
  L.bag_of = take(4 * (size_t)N);
  L.bag_sorted = take(4 * (size_t)N);
  L.psw_sorted = take(4 * (size_t)N);
  L.coef = take(p.pooling == TBE_POOL_MEAN ? 4 * (size_t)N : 0);
  L.run_starts = take(4 * (size_t)(N + 1));
  L.run_table = take(4 * (size_t)N);
  L.long_list = take(16 * (size_t)L.chunk_cap);  // one record per chunk
  L.sub_list = take(8 * (size_t)L.sub_cap);
  L.gofs = take(8 * (size_t)(p.T + 1));
  L.partials = take(4 * (size_t)L.chunk_cap * L.slot_floats);
  L.zero_begin = off;  // cleared by a memset before the first kernel
  L.hist = take(4 * 4 * 256);
  L.seg_hist = take(L.seg_dbits > 0 ? 4 * (size_t)p.T * 2 * kSegBk : 0);
  L.seg_inv = take(L.seg_dbits > 0 ? 4 * (size_t)p.T : 0);
  L.sort_tiles = take(4 * 4);
  L.rle_tile = take(4);
  L.counters = take(4 * (size_t)kCntStride * kNumCounters);
  L.zero_end = off;
  L.lin_zero_begin = off;  // cleared by the linearize kernel
  L.sort_lookback = take(4 * (size_t)L.npass * L.sort_ntiles * (L.seg_dbits > 0 ? kSegBk : 256));
  L.rle_lookback = take(4 * (size_t)L.rle_ntiles * kWordStride);
  L.combine = take(4 * (size_t)L.chunk_cap);
  L.lin_zero_end = off;
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------------------
// 1. linearize + digit histograms
// ---------------------------------------------------------------------------
struct LinArgs {
  IdxPtr indices;
  IdxPtr offsets;
  const TableMeta* meta;
  uint32_t* keys;
  int32_t* bag_of;
  uint32_t* hist;      // [4][256]
  uint32_t* counters;  // kCntInvalid
  int32_t* status;
  void* zero;          // look-back words and combine counters, cleared here
  int64_t zero_words4; // ... in 16-byte words
  int64_t N;
  int32_t T, B, npass;
  uint32_t sentinel;   // total_rows
  // segmented sort (seg_dbits > 0): keys are ids within their table (an id
  // outside the table becomes rows_t), digit counts are per table
  int32_t seg_dbits;
  uint32_t* seg_hist;  // [T][2][kSegBk]
  uint32_t* seg_inv;   // [T] ids outside their table
  // mean pooling: coef[i] = (weight of lookup i, or 1) / (its bag's lookups)
  const float* psw;
  float* coef;         // null: sum pooling
};

// largest g in [lo, hi] with offsets[g] <= pos (global memory)
__device__ __forceinline__ int32_t bag_search_global(const IdxPtr& offsets, int32_t lo, int32_t hi, int64_t pos) {
  while (lo < hi) {
    int32_t mid = lo + ((hi - lo + 1) >> 1);
    if (offsets.ldg(mid) <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Largest g in [0, nb) with offsets[g] <= pos, found by one warp with a
// 32-ary search: each round the lanes probe 32 evenly spaced bags and keep
// the sub-range after the last probe that is <= pos (3 rounds for 16K bags).
// Broken (non-monotone) offsets still give an index inside [0, nb).
__device__ __forceinline__ int32_t bag_search_warp(const IdxPtr& offsets, int32_t nb, int64_t pos, int lane) {
  int32_t lo = 0, hi = nb - 1;
  while (hi > lo) {
    const int32_t step = (hi - lo + 32) / 32;  // ceil((hi - lo + 1) / 32)
    const int32_t cand = lo + lane * step;
    const bool ok = cand <= hi && offsets.ldg(cand) <= pos;
    const unsigned m = __ballot_sync(kFull, ok);
    if (m == 0) break;  // pos precedes every probe: lo
    const int last = 31 - __clz(m);
    lo = lo + last * step;
    hi = min(hi, lo + step - 1);
    if (step == 1) break;
  }
  return lo;
}

template <int IPT>
__global__ void __launch_bounds__(kLinThreads) linearize_kernel(const LinArgs a) {
  constexpr int kLinTile = kLinThreads * IPT;
  release_dependents();
  __shared__ uint32_t s_hist[4][256];
  __shared__ int64_t s_off[kLinOffs];
  __shared__ int32_t s_g0, s_ng;
  __shared__ uint32_t s_inv;
  const int tid = threadIdx.x, lane = tid & 31;
  const int32_t nb = a.T * a.B;
  for (int k = tid; k < 4 * 256; k += kLinThreads) (&s_hist[0][0])[k] = 0;
  if (tid == 0) s_inv = 0;
  // clear the look-back words and combine counters the later kernels use
  {
    const int64_t gtid = (int64_t)blockIdx.x * kLinThreads + tid;
    const int64_t gstride = (int64_t)gridDim.x * kLinThreads;
    uint4* z = reinterpret_cast<uint4*>(a.zero);
    for (int64_t k = gtid; k < a.zero_words4; k += gstride) z[k] = make_uint4(0, 0, 0, 0);
  }
  const int64_t p0 = (int64_t)blockIdx.x * kLinTile;
  const int64_t p1 = min(a.N, p0 + kLinTile);
  // all of this thread's ids are requested first (the bag search below
  // overlaps their latency)
  constexpr int kIPT = IPT;
  uint64_t id[kIPT];  // raw id bits (out of range for the table when invalid)
#pragma unroll
  for (int q = 0; q < kIPT; ++q) {
    const int64_t i = p0 + q * kLinThreads + tid;
    id[q] = i < p1 ? a.indices.id_bits(i) : 0;
  }
  if (tid < 64) {  // warp 0 finds the bag of p0, warp 1 the bag of p1 - 1
    const int32_t g = bag_search_warp(a.offsets, nb, tid < 32 ? p0 : p1 - 1, lane);
    if (tid == 0) s_g0 = g;
    if (tid == 32) s_ng = g;
  }
  __syncthreads();
  if (tid == 0) s_ng = max(s_ng - s_g0 + 1, 1);
  __syncthreads();
  const int32_t g0 = s_g0, ng = s_ng;
  const int32_t t_first = g0 / max(a.B, 1);
  const bool staged = ng <= kLinOffs;
  if (staged)
    for (int k = tid; k < ng; k += kLinThreads) s_off[k] = a.offsets.ldg(g0 + k);
  __syncthreads();
  int bad = 0, invalid = 0;
#pragma unroll
  for (int q = 0; q < kIPT; ++q) {
    const int64_t i = p0 + q * kLinThreads + tid;
    if (i >= p1) break;
    int32_t g;
    if (staged) {
      int lo = 0, hi = ng - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
      }
      g = g0 + lo;
    } else {
      g = bag_search_global(a.offsets, g0, g0 + ng - 1, i);
    }
    const int32_t t = g / a.B;
    const int32_t b = g - t * a.B;
    if (a.coef) {  // mean pooling: the lookup's share of its bag
      const int64_t len = a.offsets.ldg(g + 1) - a.offsets.ldg(g);
      const float w = (a.psw && __ldg(&a.meta[t].weighted)) ? __ldg(a.psw + i) : 1.f;
      a.coef[i] = len > 0 ? __fdiv_rn(w, (float)len) : 0.f;
    }
    const int32_t rows = __ldg(&a.meta[t].rows);
    const bool valid = id[q] < (uint64_t)rows;
    if (!valid) { bad = 1; ++invalid; }
    uint32_t key;
    if (a.seg_dbits > 0) {
      key = valid ? (uint32_t)id[q] : (uint32_t)rows;
      const uint32_t dm = (1u << a.seg_dbits) - 1u;
      if (t == t_first) {  // the block's first table is counted in shared memory
        uint32_t* sh = &s_hist[0][0];  // two 512-bucket histograms back to back
        atomicAdd(&sh[key & dm], 1u);
        atomicAdd(&sh[kSegBk + ((key >> a.seg_dbits) & dm)], 1u);
        if (!valid) atomicAdd(&s_inv, 1u);
      } else {
        atomicAdd(&a.seg_hist[(size_t)t * 2 * kSegBk + (key & dm)], 1u);
        atomicAdd(&a.seg_hist[((size_t)t * 2 + 1) * kSegBk + ((key >> a.seg_dbits) & dm)], 1u);
        if (!valid) atomicAdd(&a.seg_inv[t], 1u);
      }
    } else {
      key = valid ? (uint32_t)(__ldg(&a.meta[t].row_base) + id[q]) : a.sentinel;
      for (int p = 0; p < a.npass; ++p) atomicAdd(&s_hist[p][(key >> (8 * p)) & 0xffu], 1u);
    }
    a.keys[i] = key;
    a.bag_of[i] = b;
  }
  // offsets must start at 0, never decrease and end at N
  const int64_t gstride = (int64_t)gridDim.x * kLinThreads;
  for (int64_t g = (int64_t)blockIdx.x * kLinThreads + tid; g < nb; g += gstride) {
    const int64_t o0 = a.offsets.ldg(g), o1 = a.offsets.ldg(g + 1);
    if (o1 < o0 || (g == 0 && o0 != 0) || (g == nb - 1 && o1 != a.N)) bad |= 2;
  }
  if (bad & 1) report(a.status, TBE_DEV_BAD_INDEX);
  if (bad & 2) report(a.status, TBE_DEV_BAD_OFFSETS);
  if (invalid) atomicAdd(&a.counters[kCntInvalid * kCntStride], (uint32_t)invalid);
  __syncthreads();
  if (a.seg_dbits > 0) {  // s_hist holds the two 512-bucket histograms of t_first back to back
    for (int k = tid; k < 2 * kSegBk; k += kLinThreads) {
      const uint32_t c = (&s_hist[0][0])[k];
      if (c) atomicAdd(&a.seg_hist[(size_t)t_first * 2 * kSegBk + k], c);
    }
    if (tid == 0 && s_inv) atomicAdd(&a.seg_inv[t_first], s_inv);
  } else {
    for (int k = tid; k < a.npass * 256; k += kLinThreads) {
      const uint32_t c = (&s_hist[0][0])[k];
      if (c) atomicAdd(&a.hist[k], c);
    }
  }
}

// ---------------------------------------------------------------------------
// 2. onesweep radix pass
// ---------------------------------------------------------------------------
struct SortArgs {
  const uint32_t* keys_in;
  const int32_t* vals_in;  // nullptr: values are the positions themselves
  uint32_t* keys_out;
  int32_t* vals_out;
  const uint32_t* hist;    // [256] digit counts of this pass
  uint32_t* lookback;      // [ntiles][256]
  uint32_t* tile_counter;
  int32_t* status;
  const int32_t* bag_of;   // last pass only: bag sample index per position
  const float* psw;        // last pass only (may be null): weight per position
  int32_t* bag_sorted;     // last pass only: bag sample index per sorted lookup
  float* psw_sorted;       // last pass only: weight per sorted lookup
  int32_t N;
  int32_t shift;
};

template <int IPT>
__global__ void __launch_bounds__(kSortThreads, 4) sort_pass_kernel(const SortArgs a) {
  constexpr int kSortIPT = IPT;
  constexpr int kSortTile = kSortThreads * IPT;
  __shared__ uint32_t s_wcnt[kSortWarps][256];
  __shared__ uint32_t s_cnt[256];     // tile count of each digit
  __shared__ uint32_t s_start[256];   // tile-local first slot of each digit
  __shared__ int32_t s_gbase[256];    // global position of slot 0 of each digit, minus s_start
  __shared__ uint32_t s_keys[kSortTile];
  __shared__ int32_t s_vals[kSortTile];
  __shared__ uint32_t s_scan[kSortWarps];
  __shared__ int32_t s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the tile counter was cleared before the first kernel of the backward, so
  // the tile is claimed while the previous pass drains
  if (tid == 0) s_tile = (int32_t)atomicAdd(a.tile_counter, 1u);
  wait_predecessor();
  release_dependents();
  for (int k = tid; k < kSortWarps * 256; k += kSortThreads) (&s_wcnt[0][0])[k] = 0;
  s_cnt[tid] = 0;
  __syncthreads();
  const int32_t tile = s_tile;
  const int32_t wbase = tile * kSortTile + warp * (32 * kSortIPT);

  uint32_t key[kSortIPT];
  int32_t val[kSortIPT];
  uint32_t rank[kSortIPT];
#pragma unroll
  for (int k = 0; k < kSortIPT; ++k) {
    const int32_t idx = wbase + k * 32 + lane;
    const bool ok = idx < a.N;
    key[k] = ok ? __ldg(a.keys_in + idx) : 0u;
    val[k] = ok ? (a.vals_in ? __ldg(a.vals_in + idx) : idx) : 0;
  }
  // the tile's digit counts come first and are published at once, so later
  // tiles find them in their look-back without waiting for this tile's ranking
#pragma unroll
  for (int k = 0; k < kSortIPT; ++k)
    if (wbase + k * 32 + lane < a.N) atomicAdd(&s_cnt[(key[k] >> a.shift) & 0xffu], 1u);
  __syncthreads();
  uint32_t* my_word = a.lookback + (size_t)tile * 256 + tid;
  st_relaxed(my_word, (tile == 0 ? kFlagInc : kFlagAgg) | s_cnt[tid]);
  // stable rank inside the warp: items are ordered (k, lane)
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int k = 0; k < kSortIPT; ++k) {
    const int32_t idx = wbase + k * 32 + lane;
    const uint32_t d = idx < a.N ? ((key[k] >> a.shift) & 0xffu) : 256u;
    const uint32_t peers = __match_any_sync(kFull, d);
    uint32_t before = 0;
    if (d < 256) before = s_wcnt[warp][d];
    __syncwarp();
    if (d < 256) {
      rank[k] = before + __popc(peers & lt_mask);
      if ((peers & lt_mask) == 0) s_wcnt[warp][d] = before + __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();
  // per digit: warp-exclusive prefixes and the tile count (thread tid = digit)
  uint32_t cnt = 0;
  {
    const int d = tid;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) {
      const uint32_t c = s_wcnt[w][d];
      s_wcnt[w][d] = cnt;
      cnt += c;
    }
  }
  // block exclusive scan of the digit counts -> s_start
  uint32_t x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_scan[warp] = x;
  // global digit base: exclusive scan of this pass's histogram
  const uint32_t h = __ldg(a.hist + tid);
  uint32_t hx = h;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, hx, o);
    if (lane >= o) hx += y;
  }
  __syncthreads();
  uint32_t wsum = 0;
  for (int w = 0; w < warp; ++w) wsum += s_scan[w];
  s_start[tid] = wsum + x - cnt;
  __syncthreads();
  // place items in tile-local sorted order (only tile-local prefixes are
  // needed, so this happens before the look-back and frees the item registers)
#pragma unroll
  for (int k = 0; k < kSortIPT; ++k) {
    const int32_t idx = wbase + k * 32 + lane;
    if (idx < a.N) {
      const uint32_t d = (key[k] >> a.shift) & 0xffu;
      const uint32_t slot = s_start[d] + s_wcnt[warp][d] + rank[k];
      s_keys[slot] = key[k];
      s_vals[slot] = val[k];
    }
  }
  if (lane == 31) s_scan[warp] = hx;
  __syncthreads();
  uint32_t hsum = 0;
  for (int w = 0; w < warp; ++w) hsum += s_scan[w];
  const uint32_t gdigit = hsum + hx - h;
  // decoupled look-back over earlier tiles for this digit: the words of up to
  // 32 predecessors are requested together (each tile owns its own 1 KB of
  // words, so no line has two writers) and summed, without branches, back to
  // the nearest inclusive one.  A window with a word not yet published goes
  // to the out-of-line slow path.
  uint32_t excl = 0;
  if (tile > 0) {
    const uint32_t* col = a.lookback + tid;
    for (int32_t hi = tile - 1; hi >= 0; hi -= 32) {
      uint32_t v[32];
      uint32_t inc = 0, miss = 0, upto = 0;
      for (int retry = 0; retry < kWindowRetries; ++retry) {  // the whole window again while words are missing
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = hi - q >= 0 ? ld_relaxed(col + (size_t)(hi - q) * 256) : kFlagInc;
        inc = 0;
        miss = 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          inc |= (v[q] >> 31) << q;
          miss |= (uint32_t)((v[q] >> 30) == 0u) << q;
        }
        upto = window_upto(inc);
        if (!(miss & upto)) break;
        __nanosleep(32);
      }
      if (miss & upto) {
        const unsigned long long r = lookback_window_slow(col, 256, hi, a.status);
        excl += (uint32_t)r;
        if (r >> 32) break;
        continue;
      }
      uint32_t sum = 0;
#pragma unroll
      for (int q = 0; q < 32; ++q) sum += ((upto >> q) & 1u) ? (v[q] & kValMask) : 0u;
      excl += sum;
      if (inc) break;
    }
    st_relaxed(my_word, kFlagInc | ((excl + cnt) & kValMask));
  }
  s_gbase[tid] = (int32_t)(gdigit + excl) - (int32_t)s_start[tid];
  __syncthreads();
  const int32_t n_tile = min(kSortTile, a.N - tile * kSortTile);
#pragma unroll
  for (int r = 0; r < IPT; ++r) {  // unrolled: the gathers of the last pass are all in flight together
    const int i = tid + r * kSortThreads;
    if (i >= n_tile) break;
    const uint32_t k = s_keys[i];
    const int32_t dst = s_gbase[(k >> a.shift) & 0xffu] + i;
    if ((uint32_t)dst < (uint32_t)a.N) {  // always true unless a wait timed out
      const int32_t v = s_vals[i];
      a.keys_out[dst] = k;
      a.vals_out[dst] = v;
      if (a.bag_sorted) {  // carry each lookup's bag and weight through the same order
        a.bag_sorted[dst] = __ldg(a.bag_of + v);
        if (a.psw_sorted) a.psw_sorted[dst] = __ldg(a.psw + v);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2b. segmented radix pass (few tables of at most 2^18 rows)
// ---------------------------------------------------------------------------
// The lookups of table t are the contiguous range [offsets[t*B],
// offsets[(t+1)*B]) and their keys the contiguous range of rows of table t,
// so sorting every table's range by id sorts the whole batch.  Ids need
// fewer bits than global rows (17 instead of 20 for 8 tables of 100 K rows),
// which makes two passes of up to 9 bits enough, and a tile's look-back stops
// at the first tile of its table.  An id outside its table has key rows_t and
// sorts to the end of its table; the last pass moves those lookups behind all
// valid ones (in position order, as the global sort with its sentinel does)
// and writes the global key table_row_base[t] + id (or the sentinel).
struct SegSortArgs {
  const uint32_t* keys_in;  // ids within the table
  const int32_t* vals_in;   // nullptr: values are the positions themselves
  uint32_t* keys_out;
  int32_t* vals_out;
  const uint32_t* hist;     // [T][2][kSegBk] digit counts per table
  const uint32_t* inv;      // [T] ids outside their table
  IdxPtr offsets;
  const TableMeta* meta;
  uint32_t* lookback;       // [tiles][kSegBk] of this pass
  uint32_t* tile_counter;
  int32_t* status;
  const int32_t* bag_of;    // last pass only
  const float* psw;
  int32_t* bag_sorted;
  float* psw_sorted;
  int32_t N, T, B, pass, dbits, last;
  uint32_t sentinel;        // total_rows
};

// Inclusive scan over the 256 threads of a block (one value each); `s_w` is
// 8 words of shared scratch.  Returns the inclusive prefix, `total` gets the
// block total.  Every thread must call it.
__device__ __forceinline__ uint32_t block_scan256(uint32_t x, uint32_t* s_w, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  uint32_t before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kSortWarps; ++w) {
    const uint32_t v = s_w[w];
    before += w < warp ? v : 0u;
    total += v;
  }
  __syncthreads();  // s_w is reused by the caller's next scan
  return before + x;
}

template <int IPT>
__global__ void __launch_bounds__(kSortThreads, 2) seg_sort_pass_kernel(const SegSortArgs a) {
  constexpr int kTile = kSortThreads * IPT;
  __shared__ uint32_t s_wcnt[kSortWarps][kSegBk];
  __shared__ uint32_t s_cnt[kSegBk];    // tile count of each digit
  __shared__ uint32_t s_start[kSegBk];  // tile-local first slot of each digit
  __shared__ int32_t s_gbase[kSegBk];   // table-local position of slot 0 of each digit, minus s_start
  __shared__ uint32_t s_keys[kTile];
  __shared__ int32_t s_vals[kTile];
  __shared__ uint32_t s_w[kSortWarps];
  __shared__ int64_t s_P[kSegMaxT + 1];  // first lookup of each table
  __shared__ int32_t s_tp[kSegMaxT + 1]; // first tile of each table
  __shared__ int32_t s_ip[kSegMaxT + 1]; // ids outside their table before each table
  __shared__ int32_t s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the tile counter (cleared before the first kernel of the backward) and
  // the offsets (an input) are read while the previous kernel drains
  if (tid == 0) s_tile = (int32_t)atomicAdd(a.tile_counter, 1u);
  for (int k = tid; k < kSortWarps * kSegBk; k += kSortThreads) (&s_wcnt[0][0])[k] = 0;
  for (int k = tid; k < kSegBk; k += kSortThreads) s_cnt[k] = 0;
  // table ranges, clamped so that broken offsets still give ranges inside [0, N)
  if (tid <= a.T) {
    int64_t P = a.offsets.ldg((int64_t)tid * a.B);
    s_P[tid] = min(max(P, (int64_t)0), (int64_t)a.N);
  }
  wait_predecessor();
  release_dependents();
  __syncthreads();
  if (warp == 0) {  // tiles and invalid ids per table, two tables per lane
    int32_t nt[2], iv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = 2 * lane + h;
      const int64_t n = t < a.T ? max(s_P[t + 1] - s_P[t], (int64_t)0) : 0;
      nt[h] = (int32_t)((n + kTile - 1) / kTile);
      iv[h] = t < a.T ? (int32_t)__ldg(a.inv + t) : 0;
    }
    int32_t x = nt[0] + nt[1], y = iv[0] + iv[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t xu = __shfl_up_sync(kFull, x, o), yu = __shfl_up_sync(kFull, y, o);
      if (lane >= o) { x += xu; y += yu; }
    }
    const int32_t x0 = x - nt[0] - nt[1], y0 = y - iv[0] - iv[1];
    if (2 * lane <= a.T) { s_tp[2 * lane] = x0; s_ip[2 * lane] = y0; }
    if (2 * lane + 1 <= a.T) { s_tp[2 * lane + 1] = x0 + nt[0]; s_ip[2 * lane + 1] = y0 + iv[0]; }
  }
  __syncthreads();
  const int32_t tile = s_tile;
  if (tile >= s_tp[a.T]) return;  // more blocks are launched than tables need
  int t = 0;
  {
    int lo = 0, hi = a.T - 1;  // largest t with s_tp[t] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tp[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    t = lo;
  }
  const int32_t k = tile - s_tp[t];  // tile within the table
  const int64_t seg_lo = s_P[t];
  const int32_t n_seg = (int32_t)(s_P[t + 1] - seg_lo);
  const int32_t base = k * kTile;    // first table-local position of the tile
  const int32_t n_tile = min(kTile, n_seg - base);
  const uint32_t dmask = (1u << a.dbits) - 1u;
  const int shift = a.pass * a.dbits;

  uint32_t key[IPT];
  int32_t val[IPT];
  uint32_t rank[IPT];
  const int32_t wbase = warp * (32 * IPT);
#pragma unroll
  for (int q = 0; q < IPT; ++q) {
    const int32_t li = wbase + q * 32 + lane;
    const bool ok = li < n_tile;
    const int64_t gi = seg_lo + base + li;
    key[q] = ok ? __ldg(a.keys_in + gi) : 0u;
    val[q] = ok ? (a.vals_in ? __ldg(a.vals_in + gi) : (int32_t)gi) : 0;
  }
  // the tile's digit counts come first and are published at once, so later
  // tiles of the table find them in their look-back without waiting for this
  // tile's ranking
#pragma unroll
  for (int q = 0; q < IPT; ++q)
    if (wbase + q * 32 + lane < n_tile) atomicAdd(&s_cnt[(key[q] >> shift) & dmask], 1u);
  __syncthreads();
  uint32_t* words = a.lookback + (size_t)tile * kSegBk;
#pragma unroll
  for (int h = 0; h < 2; ++h) st_relaxed(words + tid + h * 256, (k == 0 ? kFlagInc : kFlagAgg) | s_cnt[tid + h * 256]);
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int q = 0; q < IPT; ++q) {  // stable rank inside the warp: items are ordered (q, lane)
    const int32_t li = wbase + q * 32 + lane;
    const uint32_t d = li < n_tile ? ((key[q] >> shift) & dmask) : 0xffffu;
    const uint32_t peers = __match_any_sync(kFull, d);
    uint32_t before = 0;
    if (d < kSegBk) before = s_wcnt[warp][d];
    __syncwarp();
    if (d < kSegBk) {
      rank[q] = before + __popc(peers & lt_mask);
      if ((peers & lt_mask) == 0) s_wcnt[warp][d] = before + __popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();
  // per digit (thread tid owns digits tid and tid + 256): warp-exclusive
  // prefixes and the tile count, published at once
  uint32_t cnt[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int d = tid + h * 256;
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) {
      const uint32_t v = s_wcnt[w][d];
      s_wcnt[w][d] = c;
      c += v;
    }
    cnt[h] = c;
  }
  // tile-local starts and table-local digit bases (exclusive scans over 512 digits)
  uint32_t tot0, tot1;
  const uint32_t c0 = block_scan256(cnt[0], s_w, tot0);
  const uint32_t c1 = block_scan256(cnt[1], s_w, tot1);
  s_start[tid] = c0 - cnt[0];
  s_start[tid + 256] = tot0 + c1 - cnt[1];
  const uint32_t* th = a.hist + ((size_t)t * 2 + a.pass) * kSegBk;
  const uint32_t h0 = __ldg(th + tid), h1 = __ldg(th + tid + 256);
  uint32_t ht0, ht1;
  const uint32_t g0 = block_scan256(h0, s_w, ht0) - h0;
  const uint32_t g1 = ht0 + block_scan256(h1, s_w, ht1) - h1;
  __syncthreads();  // s_start complete
#pragma unroll
  for (int q = 0; q < IPT; ++q) {  // tile-local sorted order
    const int32_t li = wbase + q * 32 + lane;
    if (li < n_tile) {
      const uint32_t d = (key[q] >> shift) & dmask;
      const uint32_t slot = s_start[d] + s_wcnt[warp][d] + rank[q];
      s_keys[slot] = key[q];
      s_vals[slot] = val[q];
    }
  }
  // look-back over the earlier tiles of this table (k of them), both digits
  // of the thread in the same 32-tile windows
  uint32_t excl[2] = {0u, 0u};
  if (k > 0) {
    bool done[2] = {false, false};
    for (int32_t back = 1; back <= k && !(done[0] && done[1]); back += 32) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (done[h]) continue;
        const uint32_t* col = a.lookback + tid + h * 256;
        const int32_t hi = tile - back;       // nearest predecessor of this window
        const int32_t lo_tile = tile - k;     // the table's first tile (inclusive word)
        uint32_t v[32];
        uint32_t inc = 0, miss = 0, upto = 0;
        for (int retry = 0; retry < kWindowRetries; ++retry) {  // the whole window again while words are missing
#pragma unroll
          for (int q = 0; q < 32; ++q)
            v[q] = hi - q >= lo_tile ? ld_relaxed(col + (size_t)(hi - q) * kSegBk) : kFlagInc;
          inc = 0;
          miss = 0;
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            inc |= (v[q] >> 31) << q;
            miss |= (uint32_t)((v[q] >> 30) == 0u) << q;
          }
          upto = window_upto(inc);
          if (!(miss & upto)) break;
          __nanosleep(32);
        }
        if (miss & upto) {
          const unsigned long long r = lookback_window_slow(col, kSegBk, hi, a.status);
          excl[h] += (uint32_t)r;
          if (r >> 32) done[h] = true;
          continue;
        }
        uint32_t sum = 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) sum += ((upto >> q) & 1u) ? (v[q] & kValMask) : 0u;
        excl[h] += sum;
        if (inc) done[h] = true;
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) st_relaxed(words + tid + h * 256, kFlagInc | ((excl[h] + cnt[h]) & kValMask));
  }
  s_gbase[tid] = (int32_t)(g0 + excl[0]) - (int32_t)s_start[tid];
  s_gbase[tid + 256] = (int32_t)(g1 + excl[1]) - (int32_t)s_start[tid + 256];
  __syncthreads();
  // scatter: table-local position s of slot i is s_gbase[digit] + i
  const int32_t n_inv_t = s_ip[t + 1] - s_ip[t];
  const int32_t n_valid_t = n_seg - n_inv_t;
  const int64_t n_valid = (int64_t)a.N - s_ip[a.T];
  const uint32_t row_base = a.last ? (uint32_t)__ldg(&a.meta[t].row_base) : 0u;
#pragma unroll
  for (int r = 0; r < IPT; ++r) {  // unrolled: the gathers of the last pass are all in flight together
    const int i = tid + r * kSortThreads;
    if (i >= n_tile) break;
    const uint32_t key_i = s_keys[i];
    const int32_t sl = s_gbase[(key_i >> shift) & dmask] + i;
    int64_t dst = seg_lo + sl;
    uint32_t kout = key_i;
    if (a.last) {  // valid lookups close up; ids outside their table go behind all of them
      if (sl < n_valid_t) {
        dst = seg_lo - s_ip[t] + sl;
        kout = row_base + key_i;
      } else {
        dst = n_valid + s_ip[t] + (sl - n_valid_t);
        kout = a.sentinel;
      }
    }
    if ((uint64_t)dst < (uint64_t)a.N && (uint32_t)sl < (uint32_t)n_seg) {  // false only for broken inputs
      const int32_t v = s_vals[i];
      a.keys_out[dst] = kout;
      a.vals_out[dst] = v;
      if (a.bag_sorted) {
        a.bag_sorted[dst] = __ldg(a.bag_of + v);
        if (a.psw_sorted) a.psw_sorted[dst] = __ldg(a.psw + v);
      }
    }
  }
}

// First row of the table after `tp` (tp = -1: the first table); no further
// table: the largest key.
__device__ __forceinline__ int64_t next_table_base(const TableMeta* meta, int32_t T, int tp) {
  return tp + 1 < T ? __ldg(&meta[tp + 1].row_base) : INT64_MAX;
}

// A run of key `key` starts at unique index u after keys of table tp: every
// table in (tp, table(key)] starts with u unique rows below it.  Returns
// table(key).
__device__ __noinline__ int cross_tables(const TableMeta* meta, int32_t T, int64_t* unique_count, int tp,
                                         int64_t key, uint32_t u) {
  const int tk = table_of_row(meta, T, key);
  for (int t = tp + 1; t <= tk; ++t) unique_count[t] = u;
  return tk;
}

// After the last valid key (table tk): the tables after it, and the end
// marker T, see all U unique rows below them.
__device__ __noinline__ void finish_tables(int64_t* unique_count, int32_t T, int tk, uint32_t U) {
  for (int t = tk + 1; t <= T; ++t) unique_count[t] = U;
}

// ---------------------------------------------------------------------------
// 3. run-length segmentation
// ---------------------------------------------------------------------------
struct RleArgs {
  const uint32_t* keys;  // sorted
  const TableMeta* meta;
  int64_t* unique_count; // [T+1] per-table prefix of the unique rows
  int32_t T;
  int64_t* unique_rows;
  int32_t* run_starts;
  int32_t* run_table;    // table of every run
  uint32_t* lookback;
  uint32_t* tile_counter;
  uint32_t* counters;
  int32_t* status;
  int32_t N;
  int32_t ntiles;
  uint32_t sentinel;
};

template <int IPT>
__global__ void __launch_bounds__(kRleThreads) rle_kernel(const RleArgs a) {
  constexpr int kRleIPT = IPT;
  constexpr int kRleTile = kRleThreads * IPT;
  __shared__ uint32_t s_scan[kRleThreads / 32];
  __shared__ uint32_t s_lb[2 * (kRleThreads / 32)];
  __shared__ uint32_t s_excl;
  __shared__ int32_t s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the tile counter was cleared before the first kernel of the backward
  if (tid == 0) s_tile = (int32_t)atomicAdd(a.tile_counter, 1u);
  wait_predecessor();
  release_dependents();
  __syncthreads();
  const int32_t tile = s_tile;
  const int32_t j0 = tile * kRleTile + tid * kRleIPT;
  uint32_t k[kRleIPT];
  // the key before and the key after this thread's keys are requested with them
  uint32_t prev = (j0 > 0 && j0 - 1 < a.N) ? __ldg(a.keys + j0 - 1) : 0xffffffffu;
  const uint32_t knext = (j0 + kRleIPT < a.N) ? __ldg(a.keys + j0 + kRleIPT) : a.sentinel;
  int64_t prevk = (j0 > 0 && j0 - 1 < a.N) ? (int64_t)prev : -1;
  if (prevk >= (int64_t)a.sentinel) prevk = -1;
  uint32_t flags = 0, nflag = 0;
#pragma unroll
  for (int q = 0; q < kRleIPT; ++q) {
    const int32_t j = j0 + q;
    k[q] = j < a.N ? __ldg(a.keys + j) : a.sentinel;
    const bool f = j < a.N && k[q] < a.sentinel && (j == 0 || k[q] != prev);
    prev = k[q];
    flags |= (uint32_t)f << q;
    nflag += f;
  }
  // table of the key before this thread's keys and the next table's first
  // row (their loads overlap the look-back below)
  int tp = prevk < 0 ? -1 : table_of_row(a.meta, a.T, prevk);
  int64_t next_base = next_table_base(a.meta, a.T, tp);
  uint32_t x = nflag;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_scan[warp] = x;
  __syncthreads();
  uint32_t wsum = 0, total = 0;
  for (int w = 0; w < kRleThreads / 32; ++w) {
    if (w < warp) wsum += s_scan[w];
    total += s_scan[w];
  }
  const uint32_t mine = wsum + x - nflag;
  {
    uint32_t* my = a.lookback + (size_t)tile * kWordStride;
    if (tid == 0) st_relaxed(my, (tile == 0 ? kFlagInc : kFlagAgg) | total);
    const uint32_t excl = tile > 0 ? lookback_block<kRleThreads>(a.lookback, tile, a.status, s_lb) : 0u;
    if (tid == 0) {
      if (tile > 0) st_relaxed(my, kFlagInc | ((excl + total) & kValMask));
      s_excl = excl;
    }
  }
  if (tid == 0) {
    const uint32_t excl = s_excl;
    if (tile == a.ntiles - 1) {
      const uint32_t U = min(excl + total, (uint32_t)a.N);
      const uint32_t n_valid = (uint32_t)a.N - a.counters[kCntInvalid * kCntStride];
      a.counters[kCntU * kCntStride] = U;
      a.run_starts[U] = (int32_t)n_valid;
    }
  }
  __syncthreads();
  uint32_t u = s_excl + mine;
  // per-table counts: unique_count[t] = number of unique rows below
  // table_row_base[t].  A run start whose key lies past the table of the
  // previous valid key writes the count for every table boundary in between;
  // the last valid key writes U for the tables after it.  The thread tracks
  // the table of its latest key and the next table's first row, so the
  // search for a key's table only runs at a boundary (out of line).
  if (j0 == 0 && (a.N == 0 || k[0] >= a.sentinel))  // no valid lookup at all
    for (int t = 0; t <= a.T; ++t) a.unique_count[t] = 0;
#pragma unroll
  for (int q = 0; q < kRleIPT; ++q) {
    const int32_t j = j0 + q;
    if ((flags & (1u << q)) && u < (uint32_t)a.N) {  // u < N unless a wait timed out
      a.unique_rows[u] = (int64_t)k[q];
      a.run_starts[u] = j;
      if ((int64_t)k[q] >= next_base) {
        tp = cross_tables(a.meta, a.T, a.unique_count, tp, (int64_t)k[q], u);
        next_base = next_table_base(a.meta, a.T, tp);
      }
      a.run_table[u] = tp;
      ++u;
    }
    const uint32_t nk = q + 1 < kRleIPT ? k[q + 1] : knext;
    if (j < a.N && k[q] < a.sentinel && (j == a.N - 1 || nk >= a.sentinel))  // last valid key
      finish_tables(a.unique_count, a.T, tp, min(u, (uint32_t)a.N));
  }
}

// ---------------------------------------------------------------------------
// 4. classify runs; per-table run counts and row-gradient offsets
// ---------------------------------------------------------------------------
struct ClsArgs {
  const int64_t* unique_rows;
  const int32_t* run_starts;
  const TableMeta* meta;
  int4* long_list;          // per chunk: {run u, its first chunk, chunks, length}
  unsigned long long* long_counter;  // (runs << 32) | chunks
  uint32_t* counters;
  int2* sub_list;           // short-run work items {batch, part}
  const int64_t* unique_count;  // [T+1], written by the segmentation kernel
  int64_t* gofs;            // [T+1] float offset of each table's block
  int32_t* status;
  int64_t capacity;
  int32_t T;
  int32_t tau;
  int32_t chunk;
  int32_t item_lookups;     // lookups per short-run work item (>= tau)
};

__global__ void __launch_bounds__(kClsThreads) classify_kernel(const ClsArgs a) {
  wait_predecessor();
  release_dependents();
  __shared__ uint32_t s_scan[3][kClsThreads / 32];
  __shared__ unsigned long long s_base;
  __shared__ uint32_t s_sub_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t U = (int32_t)a.counters[kCntU * kCntStride];
  if (blockIdx.x == 0) {
    // float offset of each table's block of row gradients:
    // gofs[t] = sum_{t' < t} (unique rows of t') * D_t'
    const int per = (a.T + kClsThreads - 1) / kClsThreads;
    int64_t mine = 0;
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) mine += (a.unique_count[t + 1] - a.unique_count[t]) * (int64_t)__ldg(&a.meta[t].D);
    }
    __shared__ int64_t s_part[kClsThreads / 32];
    int64_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    int64_t run = x - mine;
    for (int w = 0; w < warp; ++w) run += s_part[w];
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) {
        a.gofs[t] = run;
        run += (a.unique_count[t + 1] - a.unique_count[t]) * (int64_t)__ldg(&a.meta[t].D);
      }
    }
    if (tid == kClsThreads - 1) {
      a.gofs[a.T] = run;
      if (run > a.capacity) report(a.status, TBE_DEV_CAPACITY);
    }
    __syncthreads();
  }
  const int32_t stride = gridDim.x * kClsThreads;
  for (int32_t u0 = blockIdx.x * kClsThreads; u0 < U; u0 += stride) {
    const int32_t u = u0 + tid;
    int32_t len = 0;
    if (u < U) len = a.run_starts[u + 1] - a.run_starts[u];
    const bool is_long = u < U && len >= a.tau;
    const uint32_t nch = is_long ? (uint32_t)((len + a.chunk - 1) / a.chunk) : 0u;
    // this warp's 32 runs are one batch; its short lookups are cut into
    // parts of item_lookups each (one work item per part)
    uint32_t short_sum = (u < U && !is_long) ? (uint32_t)len : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) short_sum += __shfl_xor_sync(kFull, short_sum, o);
    const uint32_t nsub = (short_sum + a.item_lookups - 1) / a.item_lookups;
    uint32_t x0 = is_long, x1 = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y0 = __shfl_up_sync(kFull, x0, o), y1 = __shfl_up_sync(kFull, x1, o);
      if (lane >= o) { x0 += y0; x1 += y1; }
    }
    if (lane == 31) { s_scan[0][warp] = x0; s_scan[1][warp] = x1; s_scan[2][warp] = nsub; }
    __syncthreads();
    uint32_t w0 = 0, w1 = 0, w2 = 0, t0 = 0, t1 = 0, t2 = 0;
    for (int w = 0; w < kClsThreads / 32; ++w) {
      if (w < warp) { w0 += s_scan[0][w]; w1 += s_scan[1][w]; w2 += s_scan[2][w]; }
      t0 += s_scan[0][w];
      t1 += s_scan[1][w];
      t2 += s_scan[2][w];
    }
    if (tid == 0 && t0 > 0)
      s_base = atomicAdd(a.long_counter, ((unsigned long long)t0 << 32) | (unsigned long long)t1);
    if (tid == 32 && t2 > 0) s_sub_base = atomicAdd(&a.counters[kCntSub * kCntStride], t2);
    __syncthreads();
    if (is_long) {  // every chunk of the run gets the run's record, so a chunk finds its run in one load
      const uint32_t cpos = (uint32_t)(s_base & 0xffffffffu) + w1 + x1 - nch;
      const int4 rec = make_int4(u, (int)cpos, (int)nch, len);
      for (uint32_t k = 0; k < nch; ++k) a.long_list[cpos + k] = rec;
    }
    for (uint32_t k = lane; k < nsub; k += 32)
      a.sub_list[s_sub_base + w2 + k] = make_int2((u0 >> 5) + warp, (int)k);
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// 5. reduce: long-run chunks (with the last-arriver combine) and short runs
// ---------------------------------------------------------------------------
struct RedArgs {
  const float* grad_out;
  const TableMeta* meta;
  const int32_t* bag_sorted;  // bag sample index of every sorted lookup
  const float* psw_sorted;    // weight of every sorted lookup (null: unweighted)
  int32_t coef_all;           // psw_sorted holds a coefficient for every table's lookups (mean pooling)
  const int64_t* unique_rows;
  const int32_t* run_starts;
  const int32_t* run_table;
  const int4* long_list;
  const unsigned long long* long_counter;
  uint32_t* counters;
  uint32_t* combine;
  float* partials;
  const int64_t* unique_count;
  const int64_t* gofs;
  float* row_grads;
  int32_t* status;
  const int2* sub_list;       // short-run work items {batch, part}
  int64_t capacity;
  int32_t T, B, sumD, tau, chunk, slot_floats, item_lookups;
  // fused exact optimizer (tbe_backward_update): every finished row gradient
  // updates its table row (and momentum) in place instead of being stored
  uint8_t* weights;
  float* momentum;
  float lr, eps;
};

// Where run u's row gradient goes and how wide it is.
struct RunInfo {
  int64_t out_off;   // float offset in row_grads
  int32_t col_off;   // first grad_out column of its table
  int32_t D;
  int32_t weighted;
  int32_t t;         // its table
};

// Per-table row-gradient offsets and unique-row counts staged in shared
// memory by every reduce block when the batch has at most kRedSmemT tables
// (one dependent global load less per work item).
constexpr int kRedSmemT = 256;
__shared__ int64_t s_red_gofs[kRedSmemT + 1];
__shared__ int64_t s_red_uc[kRedSmemT + 1];

__device__ __forceinline__ RunInfo run_info(const RedArgs& a, int32_t u) {
  const int32_t t = a.run_table[u];
  RunInfo r;
  r.t = t;
  r.D = __ldg(&a.meta[t].D);
  r.col_off = __ldg(&a.meta[t].col_off);
  r.weighted = (a.psw_sorted != nullptr) && (a.coef_all || __ldg(&a.meta[t].weighted));
  const bool staged = a.T <= kRedSmemT;
  const int64_t go = staged ? s_red_gofs[t] : a.gofs[t];
  const int64_t uc = staged ? s_red_uc[t] : a.unique_count[t];
  r.out_off = go + (int64_t)(u - uc) * r.D;
  return r;
}

// Accumulator of one lane: one float4 column chunk, two interleaved sets
// (successive lookups alternate between them, halving the serial depth).
struct Acc {
  float4 v[2];
  __device__ __forceinline__ void zero() {
    v[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    v[1] = v[0];
  }
  template <bool W>
  __device__ __forceinline__ void add(int s, float4 g, float w) {
    // weighted: the product is rounded to fp32, then added
    if (W) {
      mul2(g.x, g.y, w);
      mul2(g.z, g.w, w);
    }
    add2(v[s].x, v[s].y, g.x, g.y);
    add2(v[s].z, v[s].w, g.z, g.w);
  }
  __device__ __forceinline__ float4 sum() const {
    return make_float4(__fadd_rn(v[0].x, v[1].x), __fadd_rn(v[0].y, v[1].y), __fadd_rn(v[0].z, v[1].z),
                       __fadd_rn(v[0].w, v[1].w));
  }
};

// acc += w * g (weighted: the product is rounded to fp32, then added)
template <bool W>
__device__ __forceinline__ void add_slice(float4& acc, float4 g, float w) {
  if (W) {
    mul2(g.x, g.y, w);
    mul2(g.z, g.w, w);
  }
  add2(acc.x, acc.y, g.x, g.y);
  add2(acc.z, acc.w, g.z, g.w);
}

// Fused exact optimizer ([FBT] "Why the backward is the hard half": the
// update runs once per distinct row on its finished gradient).  OPT is 0 (no
// update: row gradients are stored), TBE_OPT_EXACT_SGD + 1 or
// TBE_OPT_EXACT_ROWWISE_ADAGRAD + 1.  Rows have at most 128 columns, so lane
// c holds columns 4c .. 4c + 3 of a row gradient (zero past the row).  The
// arithmetic is the update kernel's, so fused and separate steps agree bit
// for bit.

// Weights of global row `row` of table t: row bytes and dtype.
__device__ __forceinline__ uint8_t* weight_row(const RedArgs& a, int t, int64_t row, int& dt) {
  const TableMeta* m = a.meta + t;
  dt = __ldg(&m->dtype);
  const int64_t id = row - __ldg(&m->row_base);
  return a.weights + __ldg(&m->w_off) + id * (int64_t)__ldg(&m->D) * (dt == TBE_F32 ? 4 : 2);
}

// Updates one row from its gradient (lane quads); all lanes call it.
template <int OPT>
__device__ __forceinline__ void update_row(const RedArgs& a, int t, int64_t row, float4 g, int lane) {
  int dt;
  uint8_t* w = weight_row(a, t, row, dt);
  const int D = __ldg(&a.meta[t].D);
  const bool live = lane * 4 < D;
  const size_t qb = (size_t)lane * (dt == TBE_F32 ? 16 : 8);
  float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (live) wv = load_quad(dt, w + qb);
  float step = a.lr;
  if (OPT == TBE_OPT_EXACT_ROWWISE_ADAGRAD + 1) {
    const float m_old = a.momentum[row];
    const float ss = warp_sum(sum_sq(g, 0.f));
    float m_new = 0.f;
    step = adagrad_step(a.lr, a.eps, m_old, ss, D, &m_new);
    __syncwarp();  // every lane has read the old momentum
    if (lane == 0) a.momentum[row] = m_new;
  }
  if (live) store_quad(dt, w + qb, fma_quad(step, g, wv));
}

// Rows finished by the short-run tier wait in a per-warp shared-memory
// buffer: their gradient (lane quads) and their weights, which the lanes
// start copying (cp.async) the moment the row is finished, so the copy runs
// while the warp reduces the next runs.  Once at least kPendFlush rows wait
// (checked after every UNR <= kPendFlush lookups, so at most
// 2 * kPendFlush - 1 ever wait) they are updated from shared memory and
// stored; nothing is loaded from global memory at that point.
constexpr int kPendFlush = 4;
constexpr int kPend = 2 * kPendFlush;

struct PendRow {
  uint8_t* w;     // the row's weights
  int64_t row;    // global row (momentum index)
  float m;        // its momentum before the step (row-wise Adagrad)
  int32_t dt, D;
};

template <int OPT>
__device__ __forceinline__ void update_pending(const RedArgs& a, const float4* pend_g, const uint4* pend_w,
                                               const PendRow* pend, int n, int lane) {
  asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's weight copies have landed
#pragma unroll 1
  for (int r = 0; r < n; ++r) {
    const PendRow pr = pend[r];
    const float4 g = pend_g[r * 32 + lane];
    const uint4 raw = pend_w[r * 32 + lane];
    const bool live = lane * 4 < pr.D;
    const float4 wv = load_quad(pr.dt, reinterpret_cast<const uint8_t*>(&raw));
    float step = a.lr;
    if (OPT == TBE_OPT_EXACT_ROWWISE_ADAGRAD + 1) {
      const float ss = warp_sum(sum_sq(g, 0.f));
      float m_new = 0.f;
      step = adagrad_step(a.lr, a.eps, pr.m, ss, pr.D, &m_new);
      if (lane == 0) a.momentum[pr.row] = m_new;
    }
    if (live) store_quad(pr.dt, pr.w + (size_t)lane * (pr.dt == TBE_F32 ? 16 : 8), fma_quad(step, g, wv));
  }
}

__device__ __forceinline__ float4 ld_grad(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

constexpr int kColsPerPass = 128;      // 32 lanes x one float4

__device__ __forceinline__ int32_t clamp_bag(int32_t b, int32_t B) {
  return (uint32_t)b < (uint32_t)B ? b : 0;  // defensive: b < B always holds for valid inputs
}

__device__ __forceinline__ void store_col(float* dst, const float4& v, int c, int C4, int64_t limit_floats,
                                          int64_t dst_off) {
  if (c < C4 && dst_off + 4 * c + 4 <= limit_floats) *reinterpret_cast<float4*>(dst + dst_off + 4 * c) = v;
}

// Bag and weight of sorted lookup j (lanes past the end get bag 0, weight 1).
// `weighted`: the lookup's table uses per-sample weights (otherwise w = 1).
template <bool W>
__device__ __forceinline__ void fetch_lookup(const RedArgs& a, int32_t j, bool ok, bool weighted, int32_t& b,
                                             float& w) {
  b = 0;
  w = 1.f;
  if (ok) {
    b = clamp_bag(__ldg(a.bag_sorted + j), a.B);
    if (W && weighted) w = __ldg(a.psw_sorted + j);
  }
}

// Sum of sorted lookups [j0, j1) of one run (columns [cb, cb + 128)).  The
// bags of the next 32 lookups are requested while the current 32 gradient
// slices are in flight.
template <bool W, int UNR>
__device__ void sum_lookups(const RedArgs& a, const RunInfo& r, int32_t j0, int32_t j1, int cb, int lane,
                            Acc& acc) {
  const int C4 = r.D >> 2;
  const int c = (cb >> 2) + lane;
  const float* gcol = a.grad_out + r.col_off + 4 * c;
  int32_t nxt_b;
  float nxt_w;
  fetch_lookup<W>(a, j0 + lane, j0 + lane < j1, r.weighted, nxt_b, nxt_w);
  for (int32_t jb = j0; jb < j1; jb += 32) {
    const int n = min(32, j1 - jb);
    const int32_t my_b = nxt_b;
    const float my_w = nxt_w;
    fetch_lookup<W>(a, jb + 32 + lane, jb + 32 + lane < j1, r.weighted, nxt_b, nxt_w);
#pragma unroll 1
    for (int q0 = 0; q0 < n; q0 += UNR) {
      float4 g[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int q = q0 + u;
        const int32_t b = __shfl_sync(kFull, my_b, q & 31);
        g[u] = (q < n && c < C4) ? ld_grad(gcol + (int64_t)b * a.sumD) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) acc.add<W>(u & 1, g[u], W ? __shfl_sync(kFull, my_w, (q0 + u) & 31) : 1.f);
    }
  }
}

// One chunk of a long run.  Its partial sum (all columns) goes to its own
// workspace slot; then, level by level of a fan-in-32 tree, the chunk that
// finishes last at a node (it sees the node's arrival counter reach
// children-1 after a device-scope fence) sums the children in index order
// and writes the node's slot, or the row gradient at the root.  The order of
// every sum is fixed, so the result does not depend on arrival order.
template <bool W, int UNR, int OPT>
__device__ void long_chunk(const RedArgs& a, int32_t item, int lane) {
  const int4 rec = a.long_list[item];  // the record of the chunk's run
  const int32_t u = rec.x, e0 = rec.y, nch = rec.z, len = rec.w;
  const int32_t k = item - e0;
  const RunInfo r = run_info(a, u);
  const int32_t rs = a.run_starts[u];
  const int32_t j0 = rs + k * a.chunk, j1 = min(rs + len, j0 + a.chunk);
  const int C4 = r.D >> 2;
  for (int cb = 0; cb < r.D; cb += kColsPerPass) {
    Acc acc;
    acc.zero();
    sum_lookups<W, UNR>(a, r, j0, j1, cb, lane, acc);
    const float4 v = acc.sum();
    const int c = (cb >> 2) + lane;
    if (nch == 1) {
      if (OPT) update_row<OPT>(a, r.t, a.unique_rows[u], v, lane);  // a one-chunk run is finished here
      else store_col(a.row_grads, v, c, C4, a.capacity, r.out_off);
    } else
      store_col(a.partials + (int64_t)(e0 + k) * a.slot_floats, v, c, C4, (int64_t)1 << 62, 0);
  }
  if (nch == 1) return;
  int32_t node = k, span = 1, nodes = nch, cbase = e0;
  while (true) {
    const int32_t parent = node / kFanIn;
    const int32_t pnodes = (nodes + kFanIn - 1) / kFanIn;
    const int32_t nchild = min(kFanIn, nodes - parent * kFanIn);
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(a.combine + cbase + parent, 1u);
    old = __shfl_sync(kFull, old, 0);
    if (old != (uint32_t)(nchild - 1)) return;  // another child is still running
    __threadfence();
    const int32_t pspan = span * kFanIn;
    for (int cb = 0; cb < r.D; cb += kColsPerPass) {
      const int c = (cb >> 2) + lane;
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < C4) {
        for (int ch = 0; ch < nchild; ++ch) {
          const float* cs = a.partials + (int64_t)(e0 + (parent * kFanIn + ch) * span) * a.slot_floats;
          const float4 x = __ldcg(reinterpret_cast<const float4*>(cs + 4 * c));
          s.x = __fadd_rn(s.x, x.x);
          s.y = __fadd_rn(s.y, x.y);
          s.z = __fadd_rn(s.z, x.z);
          s.w = __fadd_rn(s.w, x.w);
        }
      }
      if (pnodes == 1) {
        if (OPT) update_row<OPT>(a, r.t, a.unique_rows[u], s, lane);  // the root: the run's gradient is finished
        else store_col(a.row_grads, s, c, C4, a.capacity, r.out_off);
      } else
        store_col(a.partials + (int64_t)(e0 + parent * pspan) * a.slot_floats, s, c, C4, (int64_t)1 << 62, 0);
    }
    if (pnodes == 1) return;  // root written: the row gradient is complete
    span = pspan;
    cbase += pnodes;  // counters of the next level follow this level's
    node = parent;
    nodes = pnodes;
  }
}

// Part `part` of a batch of 32 consecutive runs.  The short runs of the batch
// form one flattened stream of lookups in run order (lane l holds the
// metadata of run 32*batch + l); part k takes the runs whose first lookup
// falls in [k*L, (k+1)*L) of that stream (L = a.item_lookups >= the
// threshold, so no part is empty and each has fewer than L + threshold
// lookups).  The warp reduces the part's stream and stores a run's row
// gradient at its last lookup.  Long runs are skipped (their chunks are
// separate work items).
template <bool W, int UNR, int OPT>
__device__ void short_batch(const RedArgs& a, int32_t batch, int32_t part, int32_t U, int lane, float4* pend_g,
                            uint4* pend_w, PendRow* pend) {
  const int32_t u = batch * 32 + lane;
  int32_t rs = 0, len = 0;
  // fused update: global row, weights, dtype and old momentum of run u
  int64_t run_row = 0;
  uint8_t* run_wrow = nullptr;
  int32_t run_dt = TBE_F32;
  float run_m = 0.f;
  RunInfo r{0, 0, 4, 0, 0};
  if (u < U) {
    rs = a.run_starts[u];
    len = a.run_starts[u + 1] - rs;
    r = run_info(a, u);
    if (OPT) {
      run_row = a.unique_rows[u];
      run_wrow = weight_row(a, r.t, run_row, run_dt);
      if (OPT == TBE_OPT_EXACT_ROWWISE_ADAGRAD + 1) run_m = a.momentum[run_row];
    }
  }
  int npend = 0;  // rows waiting in pend (fused update)
  int32_t cnt = (u < U && len < a.tau) ? len : 0;
  {  // keep the runs of this part
    int32_t x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    const int64_t first = (int64_t)(x - cnt);
    const int64_t lo = (int64_t)part * a.item_lookups;
    if (first < lo || first >= lo + a.item_lookups) cnt = 0;
  }
  int32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const int32_t excl = incl - cnt;
  const int32_t total = __shfl_sync(kFull, incl, 31);
  if (total == 0) return;
  // do all runs of the part belong to one table?  (then every lookup shares
  // the column offset and width)
  const unsigned act = __ballot_sync(kFull, cnt > 0);
  const int first = __ffs(act) - 1;
  const int32_t coff0 = __shfl_sync(kFull, r.col_off, first);
  const int32_t D0 = __shfl_sync(kFull, r.D, first);
  const bool one_table = __all_sync(kFull, cnt == 0 || (r.col_off == coff0 && r.D == D0));
  int maxD = cnt > 0 ? r.D : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxD = max(maxD, __shfl_xor_sync(kFull, maxD, o));
  // float4 columns this run's row gradient may store (0: over capacity)
  const int32_t st_c4 = (cnt > 0 && r.out_off + r.D <= a.capacity) ? (r.D >> 2) : 0;

  for (int cb = 0; cb < maxD; cb += kColsPerPass) {
    const int c = (cb >> 2) + lane;
    // one accumulator: short runs are short chains of additions
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // run, bag and weight of flattened lookup f = fb + lane, and whether it
    // is the last lookup of its run
    auto fetch = [&](int32_t fb, int& my_r, int32_t& my_b, float& my_w, bool& my_end) {
      const int32_t f = fb + lane;
      my_r = 0;  // number of runs whose inclusive count is <= f (binary lifting)
#pragma unroll
      for (int step = 16; step > 0; step >>= 1)
        if (__shfl_sync(kFull, incl, my_r + step - 1) <= f) my_r += step;
      my_r = min(my_r, 31);
      const int32_t j = __shfl_sync(kFull, rs, my_r) + (f - __shfl_sync(kFull, excl, my_r));
      const int32_t r_incl = __shfl_sync(kFull, incl, my_r);  // every lane takes part in the shuffle
      my_end = (f < total) && (f == r_incl - 1);
      const bool wt = __shfl_sync(kFull, r.weighted, my_r) != 0;
      fetch_lookup<W>(a, j, f < total, wt, my_b, my_w);
    };
    int nxt_r;
    int32_t nxt_b;
    float nxt_w;
    bool nxt_end;
    fetch(0, nxt_r, nxt_b, nxt_w, nxt_end);
    for (int32_t fb = 0; fb < total; fb += 32) {
      const int n = min(32, total - fb);
      const int my_r = nxt_r;
      const int32_t my_b = nxt_b;
      const float my_w = nxt_w;
      const unsigned ends = __ballot_sync(kFull, nxt_end);
      if (fb + 32 < total) fetch(fb + 32, nxt_r, nxt_b, nxt_w, nxt_end);
      // lookup q ends its run: store the run's row gradient
      auto flush = [&](int q) {
        const int rr = __shfl_sync(kFull, my_r, q);
        if (OPT) {  // park the finished gradient and start copying the row's weights
          const int64_t row = __shfl_sync(kFull, run_row, rr);
          const unsigned long long wbits = __shfl_sync(kFull, (unsigned long long)(uintptr_t)run_wrow, rr);
          uint8_t* w = (uint8_t*)(uintptr_t)wbits;
          const int32_t dt = __shfl_sync(kFull, run_dt, rr);
          const int32_t D = __shfl_sync(kFull, r.D, rr);
          const float m = __shfl_sync(kFull, run_m, rr);
          pend_g[npend * 32 + lane] = acc;
          if (lane * 4 < D) {
            const uint32_t dst = smem_u32(pend_w + npend * 32 + lane);
            if (dt == TBE_F32)
              cp_async16(dst, w + (size_t)lane * 16);
            else
              asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(w + (size_t)lane * 8) : "memory");
          }
          cp_commit();
          if (lane == 0) pend[npend] = PendRow{w, row, m, dt, D};
          ++npend;
        } else {
          const int64_t off = __shfl_sync(kFull, r.out_off, rr);
          const int32_t c4 = __shfl_sync(kFull, st_c4, rr);
          if (c < c4) *reinterpret_cast<float4*>(a.row_grads + off + 4 * c) = acc;
        }
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
      };
#pragma unroll 2
      for (int q0 = 0; q0 < n; q0 += UNR) {
        float4 g[UNR];
#pragma unroll
        for (int uu = 0; uu < UNR; ++uu) {
          const int q = q0 + uu;
          const int32_t b = __shfl_sync(kFull, my_b, q & 31);
          int32_t coff = coff0, C4 = D0 >> 2;
          if (!one_table) {  // uniform branch: the lookup's own table
            const int rr = __shfl_sync(kFull, my_r, q & 31);
            coff = __shfl_sync(kFull, r.col_off, rr);
            C4 = __shfl_sync(kFull, r.D, rr) >> 2;
          }
          g[uu] = (q < n && c < C4) ? ld_grad(a.grad_out + (int64_t)b * a.sumD + coff + 4 * c)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int uu = 0; uu < UNR; ++uu) {
          add_slice<W>(acc, g[uu], W ? __shfl_sync(kFull, my_w, (q0 + uu) & 31) : 1.f);
          if ((ends >> (q0 + uu)) & 1u) flush(q0 + uu);
        }
        if (OPT && npend >= kPendFlush) {  // UNR <= kPendFlush lookups ended at most that many runs
          __syncwarp();
          update_pending<OPT>(a, pend_g, pend_w, pend, npend, lane);
          __syncwarp();  // the buffer is refilled next
          npend = 0;
        }
      }
    }
  }
  if (OPT && npend > 0) {
    __syncwarp();
    update_pending<OPT>(a, pend_g, pend_w, pend, npend, lane);
    __syncwarp();
  }
}

// UNR: grad_out slices in flight per lane; MINB: resident blocks per SM the
// register budget targets.
// Per-warp shared memory of the fused update: kPend gradients, their weights
// and their row records.
constexpr size_t kPendBytesPerWarp = (size_t)kPend * 32 * 16 * 2 + kPend * sizeof(PendRow);

template <bool W, int UNR, int MINB, int OPT>
__global__ void __launch_bounds__(kRedThreads, MINB) reduce_kernel(const RedArgs a) {
  extern __shared__ __align__(16) unsigned char red_pend[];
  float4* pend_g = reinterpret_cast<float4*>(red_pend + (threadIdx.x >> 5) * kPendBytesPerWarp);
  uint4* pend_w = reinterpret_cast<uint4*>(pend_g + kPend * 32);
  PendRow* pend = reinterpret_cast<PendRow*>(pend_w + kPend * 32);
  wait_predecessor();
  release_dependents();
  if (a.T <= kRedSmemT) {
    for (int t = threadIdx.x; t <= a.T; t += kRedThreads) {
      s_red_gofs[t] = a.gofs[t];
      s_red_uc[t] = a.unique_count[t];
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int32_t U = (int32_t)a.counters[kCntU * kCntStride];
  const int32_t n_chunks = (int32_t)(*a.long_counter & 0xffffffffu);
  const int32_t n_items = n_chunks + (int32_t)a.counters[kCntSub * kCntStride];
  // the next work item is claimed while the current one is reduced
  uint32_t claim = 0;
  if (lane == 0) claim = atomicAdd(&a.counters[kCntWork * kCntStride], 1u);
  uint32_t item = __shfl_sync(kFull, claim, 0);
  while ((int32_t)item < n_items) {
    if (lane == 0) claim = atomicAdd(&a.counters[kCntWork * kCntStride], 1u);
    if ((int32_t)item < n_chunks) {
      long_chunk<W, UNR, OPT>(a, (int32_t)item, lane);
    } else {
      const int2 rec = a.sub_list[item - n_chunks];
      short_batch<W, UNR, OPT>(a, rec.x, rec.y, U, lane, pend_g, pend_w, pend);
    }
    item = __shfl_sync(kFull, claim, 0);
  }
}

// Launch on `s` with programmatic stream serialisation: the kernel may be
// scheduled while its predecessor drains and calls wait_predecessor() before
// reading what the predecessor wrote.  Triggers stay implicit (block exit),
// so it starts only once every block of the predecessor has finished.
template <typename Arg>
int launch_pdl(void (*kernel)(Arg), int grid, int threads, cudaStream_t s, const Arg& arg, size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, arg) != cudaSuccess) return TBE_ERR_CUDA;
  return check_launch();
}

int grid_for(const void* kernel, int threads, size_t smem = 0) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
      per_sm <= 0)
    per_sm = 1;
  return per_sm * sm_count();
}

}  // namespace

size_t backward_workspace_bytes(const Plan& p, int32_t B, int64_t N) {
  return make_layout(p, B, N).total;
}

// stages: kBwdIndex (memset .. classify: everything that reads only the ids,
// offsets and per-sample weights) and/or kBwdReduce (the reduction, which
// reads grad_out); the workspace carries the index stages' results to the
// reduction, so the two may be launched separately, in order.
int launch_backward(const Plan& p, const BwdArgs& a, cudaStream_t s, int stages) {
  const int64_t N = a.N;
  if (N == 0) {
    if (stages & kBwdIndex) {
      if (cudaMemsetAsync(a.unique_count, 0, sizeof(int64_t) * (p.T + 1), s) != cudaSuccess) return TBE_ERR_CUDA;
      if (a.run_starts && cudaMemsetAsync(a.run_starts, 0, sizeof(int32_t), s) != cudaSuccess) return TBE_ERR_CUDA;
    }
    trace_mark(s, "bwd_empty");
    return TBE_OK;
  }
  const Layout L = make_layout(p, a.B, N);
  void* ws = a.workspace;
  uint32_t* counters = at<uint32_t>(ws, L.counters);
  const uint32_t sentinel = (uint32_t)p.total_rows;
  int32_t* run_starts = a.run_starts ? a.run_starts : at<int32_t>(ws, L.run_starts);
  const Tuning& tu = tuning();
  unsigned long long* long_counter = reinterpret_cast<unsigned long long*>(counters + kCntLong * kCntStride);
  if (stages & kBwdIndex) {
    if (cudaMemsetAsync(at<char>(ws, L.zero_begin), 0, L.zero_end - L.zero_begin, s) != cudaSuccess)
      return TBE_ERR_CUDA;
    trace_mark(s, "bwd_memset");

    LinArgs la;
    la.indices = a.indices;
    la.offsets = a.offsets;
    la.meta = a.meta;
    la.keys = at<uint32_t>(ws, L.keys_a);
    la.bag_of = at<int32_t>(ws, L.bag_of);
    la.hist = at<uint32_t>(ws, L.hist);
    la.counters = counters;
    la.status = a.status;
    la.zero = at<char>(ws, L.lin_zero_begin);
    la.zero_words4 = (int64_t)((L.lin_zero_end - L.lin_zero_begin) / 16);
    la.N = N;
    la.T = a.T;
    la.B = a.B;
    la.npass = L.npass;
    la.sentinel = sentinel;
    la.seg_dbits = L.seg_dbits;
    la.seg_hist = at<uint32_t>(ws, L.seg_hist);
    la.seg_inv = at<uint32_t>(ws, L.seg_inv);
    const bool mean = p.pooling == TBE_POOL_MEAN;
    la.psw = a.psw;
    la.coef = mean ? at<float>(ws, L.coef) : nullptr;
    if (L.small)
      linearize_kernel<4><<<L.lin_blocks, kLinThreads, 0, s>>>(la);
    else
      linearize_kernel<8><<<L.lin_blocks, kLinThreads, 0, s>>>(la);
    if (check_launch()) return TBE_ERR_CUDA;
    trace_mark(s, "bwd_linearize");

    int32_t* final_pos = a.sorted_positions ? a.sorted_positions : at<int32_t>(ws, L.vals_b);
    uint32_t* kin = at<uint32_t>(ws, L.keys_a);
    uint32_t* kout = at<uint32_t>(ws, L.keys_b);
    int32_t* vin = nullptr;
    int32_t* vbuf[2] = {at<int32_t>(ws, L.vals_a), at<int32_t>(ws, L.vals_b)};
    for (int pass = 0; pass < L.npass; ++pass) {
      const bool last = pass == L.npass - 1;
      int32_t* vout = last ? final_pos : vbuf[pass & 1];
      if (!last && vout == final_pos) vout = vbuf[(pass + 1) & 1];
      if (vout == vin) vout = (vin == vbuf[0]) ? vbuf[1] : vbuf[0];
      if (L.seg_dbits > 0) {
        SegSortArgs ga;
        ga.keys_in = kin;
        ga.vals_in = vin;
        ga.keys_out = kout;
        ga.vals_out = vout;
        ga.hist = at<uint32_t>(ws, L.seg_hist);
        ga.inv = at<uint32_t>(ws, L.seg_inv);
        ga.offsets = a.offsets;
        ga.meta = a.meta;
        ga.lookback = at<uint32_t>(ws, L.sort_lookback) + (size_t)pass * L.sort_ntiles * kSegBk;
        ga.tile_counter = at<uint32_t>(ws, L.sort_tiles) + pass;
        ga.status = a.status;
        ga.bag_of = at<int32_t>(ws, L.bag_of);
        ga.psw = mean ? at<float>(ws, L.coef) : a.psw;
        ga.bag_sorted = last ? at<int32_t>(ws, L.bag_sorted) : nullptr;
        ga.psw_sorted = (last && (mean || (a.psw && p.any_weighted))) ? at<float>(ws, L.psw_sorted) : nullptr;
        ga.N = (int32_t)N;
        ga.T = p.T;
        ga.B = a.B;
        ga.pass = pass;
        ga.dbits = L.seg_dbits;
        ga.last = last ? 1 : 0;
        ga.sentinel = sentinel;
        if (launch_pdl(L.small ? seg_sort_pass_kernel<6> : seg_sort_pass_kernel<12>, L.sort_ntiles, kSortThreads, s,
                       ga))
          return TBE_ERR_CUDA;
        trace_mark(s, "bwd_sort_pass");
        std::swap(kin, kout);
        vin = vout;
        continue;
      }
      SortArgs sa;
      sa.keys_in = kin;
      sa.vals_in = vin;
      sa.keys_out = kout;
      sa.vals_out = vout;
      sa.hist = at<uint32_t>(ws, L.hist) + 256 * pass;
      sa.lookback = at<uint32_t>(ws, L.sort_lookback) + (size_t)pass * L.sort_ntiles * 256;
      sa.tile_counter = at<uint32_t>(ws, L.sort_tiles) + pass;
      sa.status = a.status;
      sa.bag_of = at<int32_t>(ws, L.bag_of);
      sa.psw = mean ? at<float>(ws, L.coef) : a.psw;
      sa.bag_sorted = last ? at<int32_t>(ws, L.bag_sorted) : nullptr;
      sa.psw_sorted = (last && (mean || (a.psw && p.any_weighted))) ? at<float>(ws, L.psw_sorted) : nullptr;
      sa.N = (int32_t)N;
      sa.shift = 8 * pass;
      if (launch_pdl(L.small ? sort_pass_kernel<6> : sort_pass_kernel<12>, L.sort_ntiles, kSortThreads, s, sa))
        return TBE_ERR_CUDA;
      trace_mark(s, "bwd_sort_pass");
      std::swap(kin, kout);
      vin = vout;
    }
    const uint32_t* sorted_keys = kin;

    RleArgs ra;
    ra.keys = sorted_keys;
    ra.meta = a.meta;
    ra.unique_count = a.unique_count;
    ra.T = a.T;
    ra.unique_rows = a.unique_rows;
    ra.run_starts = run_starts;
    ra.run_table = at<int32_t>(ws, L.run_table);
    ra.lookback = at<uint32_t>(ws, L.rle_lookback);
    ra.tile_counter = at<uint32_t>(ws, L.rle_tile);
    ra.counters = counters;
    ra.status = a.status;
    ra.N = (int32_t)N;
    ra.ntiles = L.rle_ntiles;
    ra.sentinel = sentinel;
    if (launch_pdl(L.small ? rle_kernel<4> : rle_kernel<8>, L.rle_ntiles, kRleThreads, s, ra)) return TBE_ERR_CUDA;
    trace_mark(s, "bwd_rle");

    ClsArgs ca;
    ca.unique_rows = a.unique_rows;
    ca.run_starts = run_starts;
    ca.meta = a.meta;
    ca.long_list = at<int4>(ws, L.long_list);
    ca.long_counter = long_counter;
    ca.counters = counters;
    ca.unique_count = a.unique_count;
    ca.gofs = at<int64_t>(ws, L.gofs);
    ca.status = a.status;
    ca.capacity = a.row_grads_capacity;
    ca.T = a.T;
    ca.tau = tu.long_run_threshold;
    ca.chunk = L.chunk;
    ca.item_lookups = L.item_lookups;
    ca.sub_list = at<int2>(ws, L.sub_list);
    const int cls_blocks = (int)std::min<int64_t>((N + kClsThreads - 1) / kClsThreads, 4 * sm_count());
    if (launch_pdl(classify_kernel, std::max(cls_blocks, 1), kClsThreads, s, ca)) return TBE_ERR_CUDA;
    trace_mark(s, "bwd_classify");
  }
  if (!(stages & kBwdReduce)) return TBE_OK;

  RedArgs rd;
  rd.grad_out = a.grad_out;
  rd.meta = a.meta;
  rd.bag_sorted = at<int32_t>(ws, L.bag_sorted);
  rd.psw_sorted = (p.pooling == TBE_POOL_MEAN || (a.psw && p.any_weighted)) ? at<float>(ws, L.psw_sorted) : nullptr;
  rd.coef_all = p.pooling == TBE_POOL_MEAN;
  rd.unique_rows = a.unique_rows;
  rd.run_starts = run_starts;
  rd.run_table = at<int32_t>(ws, L.run_table);
  rd.long_list = at<int4>(ws, L.long_list);
  rd.long_counter = long_counter;
  rd.counters = counters;
  rd.combine = at<uint32_t>(ws, L.combine);
  rd.partials = at<float>(ws, L.partials);
  rd.unique_count = a.unique_count;
  rd.gofs = at<int64_t>(ws, L.gofs);
  rd.row_grads = a.row_grads;
  rd.status = a.status;
  rd.capacity = a.row_grads_capacity;
  rd.T = a.T;
  rd.B = a.B;
  rd.sumD = a.sumD;
  rd.tau = tu.long_run_threshold;
  rd.chunk = L.chunk;
  rd.item_lookups = L.item_lookups;
  rd.sub_list = at<int2>(ws, L.sub_list);
  rd.slot_floats = L.slot_floats;
  rd.weights = a.weights;
  rd.momentum = a.momentum;
  rd.lr = a.lr;
  rd.eps = a.eps;
  const bool weighted = rd.psw_sorted != nullptr;
  const int opt = a.opt_kind < 0 ? 0 : a.opt_kind + 1;
  const bool deep = tu.red_unroll == 8 && opt == 0;  // the fused update uses the 4-slice build
  void (*kern)(RedArgs);
  if (opt == 0)
    kern = weighted ? (deep ? reduce_kernel<true, 8, 3, 0> : reduce_kernel<true, 4, 4, 0>)
                    : (deep ? reduce_kernel<false, 8, 3, 0> : reduce_kernel<false, 4, 4, 0>);
  else if (opt == TBE_OPT_EXACT_SGD + 1)
    kern = weighted ? reduce_kernel<true, 4, 3, TBE_OPT_EXACT_SGD + 1> : reduce_kernel<false, 4, 3, TBE_OPT_EXACT_SGD + 1>;
  else
    kern = weighted ? reduce_kernel<true, 4, 3, TBE_OPT_EXACT_ROWWISE_ADAGRAD + 1>
                    : reduce_kernel<false, 4, 3, TBE_OPT_EXACT_ROWWISE_ADAGRAD + 1>;
  const size_t smem = opt ? (size_t)(kRedThreads / 32) * kPendBytesPerWarp : 0;
  static int red_grid[8][64] = {{0}};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  const int variant = opt == 0 ? (weighted ? 1 : 0) + (deep ? 2 : 0) : 4 + (weighted ? 1 : 0) + 2 * (opt - 1);
  if (red_grid[variant][dev] == 0) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TBE_ERR_CUDA;
    red_grid[variant][dev] = grid_for((const void*)kern, kRedThreads, smem);
  }
  const int64_t want = ((N + 31) / 32 + 7) / 8 + 1;
  const int rgrid = (int)std::max<int64_t>(1, std::min<int64_t>(red_grid[variant][dev], want));
  if (launch_pdl(kern, rgrid, kRedThreads, s, rd, smem)) return TBE_ERR_CUDA;
  trace_mark(s, "bwd_reduce");
  return TBE_OK;
}

}  // namespace tbe
