// tbe_forward.cu -- pooled gather-sum forward of table-batched embedding bags.
//
// [FBT] = the page "FBTriton table-batched embeddings: the backward win is a
// threshold moved from 32 to 256".
//
// What is computed ([FBT] "A lookup table that is most of the model"):
//   out[b, D_offsets[t] + c] = sum_{i in bag(t,b)} w_i * W_t[id_i, c]
// with bag (t,b) = indices[offsets[t*B+b] : offsets[t*B+b+1]], FP32
// accumulation and one round-to-nearest-even to the output type ([FBT] "The
// forward: a general gather and one clever special case").  Empty bags are
// written as zero; repeated ids are simply added again.
//
// Design (GB300): each bag is pooled by a virtual warp (VW) of `lpr` lanes,
// lpr = the power of two >= the row's 16-byte chunks, capped at a tunable
// maximum (8 by default), so a warp pools 32/lpr bags at once without any
// cross-lane reduction and every lane owns KMAX chunks of the row.  The VW
// fetches a window of 4*lpr ids of its bag with one coalesced request and
// hands them around with width-limited shuffles, then requests U rows
// (16-byte loads through the read-only path, U*KMAX chunks per lane) before
// consuming the first, keeping many independent index->row chains in flight
// (the page's "several chains" idea, widened to a whole warp).  Warp tasks
// (32/lpr bags of one table) are walked grid-stride by a grid sized to the SM
// count, and the bag bounds of a warp's next task are requested while it
// pools the current one.  Uniform layouts get a kernel specialised to their
// one dtype.
#include <algorithm>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;

__device__ __forceinline__ TableMeta load_meta(const TableMeta* p) {
  TableMeta m;
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 a = __ldg(q), b = __ldg(q + 1);
  *reinterpret_cast<uint4*>(&m) = a;
  *(reinterpret_cast<uint4*>(&m) + 1) = b;
  return m;
}

// The same, issued where it stands (the compiler may not sink it to its
// first use, behind loads that the caller waits on first).
__device__ __forceinline__ TableMeta load_meta_now(const TableMeta* p) {
  TableMeta m;
  uint4 x, y;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w) : "l"(p));
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4+16];" : "=r"(y.x), "=r"(y.y), "=r"(y.z), "=r"(y.w) : "l"(p));
  *reinterpret_cast<uint4*>(&m) = x;
  *(reinterpret_cast<uint4*>(&m) + 1) = y;
  return m;
}

constexpr int kIdsPerLane = 4;  // id window of a VW: kIdsPerLane * lpr ids

// One id window of a bag held by the lanes of its VW: lane `sub` holds ids
// base + sub + k*lpr (k < kIdsPerLane).  Ids outside the table are -1 (rows
// < 2^31, so every valid id fits 32 bits).
struct IdWin {
  int32_t id[kIdsPerLane];
  float w[kIdsPerLane];
};

template <bool WT>
__device__ __forceinline__ void load_window(const FwdArgs& a, const TableMeta& m, int lpr, int sub, int64_t base,
                                            int nwin, IdWin& iw) {
  const bool weighted = WT && m.weighted;
#pragma unroll
  for (int k = 0; k < kIdsPerLane; ++k) {  // the whole window in one request
    const int idx = k * lpr + sub;
    const uint64_t raw = idx < nwin ? a.indices.id_bits(base + idx) : 0;
    iw.id[k] = raw < (uint64_t)m.rows ? (int32_t)raw : -1;
    iw.w[k] = (weighted && idx < nwin) ? ld_stream_f32(a.psw + base + idx) : 1.f;
  }
}

// Pools bag (t, b) = [start, end) with a virtual warp of `lpr` lanes (lsh =
// log2 lpr).  Lane `sub` owns chunks sub + k*lpr (k < KMAX) of each column
// block of lpr*KMAX chunks; U rows are requested before the first is used.
template <int DT, int KMAX, int U, bool WT, typename OutT>
__device__ __forceinline__ void pool_bag(const FwdArgs& a, const TableMeta& m, int lsh, int b, int lane,
                                         int64_t start, int64_t end) {
  const int lpr = 1 << lsh;
  constexpr int E = Chunk<DT>::kElems;           // elements per chunk
  constexpr int NS = (DT == TBE_F32) ? 2 : 1;    // interleaved accumulator sets (fp32 tables)
  const int C = m.D / E;                          // chunks per row
  const int sub = lane & (lpr - 1);
  const unsigned vmask = lpr == 32 ? kFull : (((1u << lpr) - 1u) << (lane & ~(lpr - 1)));
  const char* tbl = reinterpret_cast<const char*>(a.weights) + m.w_off;
  const int64_t row_bytes = (int64_t)C * 16;
  const bool weighted = WT && m.weighted;  // WT: the call has per-sample weights
  OutT* out_row = reinterpret_cast<OutT*>(a.out) + (int64_t)b * a.sumD + m.col_off;
  const int win = kIdsPerLane * lpr;
  bool bad = false;

#pragma unroll 1
  for (int cb = 0; cb < C; cb += lpr * KMAX) {  // column blocks (wide rows only)
    float acc[NS][KMAX][E];
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[s][k][e] = 0.f;

#pragma unroll 1
    for (int64_t base = start; base < end; base += win) {
      const int nwin = (int)min((int64_t)win, end - base);
      IdWin iw;
      load_window<WT>(a, m, lpr, sub, base, nwin, iw);
#pragma unroll
      for (int slot = 0; slot < kIdsPerLane; ++slot) {  // window slot: ids slot*lpr .. slot*lpr + lpr - 1
        const int n = min(lpr, nwin - slot * lpr);
        if (n <= 0) break;
#pragma unroll 1
        for (int j0 = 0; j0 < n; j0 += U) {
          uint4 v[U][KMAX];
          float w[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int j = j0 + u;
            const int32_t id = __shfl_sync(vmask, iw.id[slot], j & (lpr - 1), lpr);
            w[u] = WT ? __shfl_sync(vmask, iw.w[slot], j & (lpr - 1), lpr) : 1.f;
            const bool live = j < n;
            const bool ok = live && id >= 0;
            bad |= live && !ok;  // reported, contributes nothing
            const char* row = tbl + (int64_t)id * row_bytes;
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
              const int c = cb + sub + k * lpr;
              v[u][k] = (ok && c < C) ? ld_row16(row + (int64_t)c * 16) : make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
              float f[E];
              Chunk<DT>::to_float(v[u][k], f);
              if (WT && weighted) {  // the product is rounded to fp32, then added
#pragma unroll
                for (int e = 0; e < E; e += 2) mul2(f[e], f[e + 1], w[u]);
              }
#pragma unroll
              for (int e = 0; e < E; e += 2) add2(acc[u % NS][k][e], acc[u % NS][k][e + 1], f[e], f[e + 1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int c = cb + sub + k * lpr;
      if (c < C) {
        float f[E];
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = NS == 2 ? __fadd_rn(acc[0][k][e], acc[NS - 1][k][e]) : acc[0][k][e];
        if (a.mean) mean_scale(f, E, end - start);
        store_out<OutT>(out_row + (int64_t)c * E, f, E, a.out_vec_ok);
      }
    }
  }
  if (bad && sub == 0) report(a.status, TBE_DEV_BAD_INDEX);
}

// One chunk per lane when the row fits the VW, else two (with column blocks
// for rows wider than 64 chunks); U = R / KMAX rows in flight.
template <int DT, int R, bool WT, typename OutT>
__device__ __forceinline__ void pool_bag_dt(const FwdArgs& a, const TableMeta& m, int lsh, int b, int lane,
                                            int64_t start, int64_t end) {
  constexpr int E = Chunk<DT>::kElems;
  if (m.D / E <= (1 << lsh))
    pool_bag<DT, 1, R, WT, OutT>(a, m, lsh, b, lane, start, end);
  else
    pool_bag<DT, 2, (R / 2 > 0 ? R / 2 : 1), WT, OutT>(a, m, lsh, b, lane, start, end);
}

// lanes per row: p = the power of two >= the row's 16-byte chunks; a VW has
// min(p, lpr_max) lanes but at least p/2 (at most two chunks per lane) and
// at most 32
__device__ __forceinline__ int lanes_per_row(const TableMeta& m, int lpr_max) {
  const int C = (m.D * (m.dtype == TBE_F32 ? 4 : 2)) >> 4;
  const int p = C <= 1 ? 1 : (1 << (32 - __clz(C - 1)));
  return min(32, max(min(p, lpr_max), p >> 1));
}

constexpr int kMaxSmemTables = TBE_MAX_TABLES;

// Work is enumerated in warp tasks: task k of table t covers bags
// b = k*G_t .. k*G_t + G_t - 1 with G_t = 32 / lanes_per_row (one bag per
// virtual warp).  Every block first builds the running task count of the
// tables in shared memory, then its warps walk the tasks grid-stride.
// DTSEL: the one table dtype of the layout, or -1 for the generic kernel.
// R: 16-byte row chunks in flight per lane.
struct Task {
  int32_t t, b, lsh;
  bool live;
};

__device__ __forceinline__ Task locate_task(const FwdArgs& a, const int32_t* s_pref, int32_t ntasks, int32_t task,
                                            int lane) {
  Task k;
  k.live = false;
  k.t = k.b = k.lsh = 0;
  if (task >= ntasks) return k;
  int lo = 0, hi = a.T - 1;  // table of this task: largest t with s_pref[t] <= task
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= task) lo = mid; else hi = mid - 1;
  }
  k.t = lo;
  k.lsh = 31 - __clz(lanes_per_row(load_meta(a.meta + lo), a.lpr_max));
  k.b = (task - s_pref[lo]) * (32 >> k.lsh) + (lane >> k.lsh);
  k.live = k.b < a.B;  // the table's last task may have idle virtual warps
  return k;
}

__device__ __forceinline__ void bag_bounds(const FwdArgs& a, const Task& k, int64_t& start, int64_t& end) {
  const int64_t g = (int64_t)k.t * a.B + k.b;
  start = a.offsets.stream(g);
  end = a.offsets.stream(g + 1);
}

// Offsets must start at 0, never decrease and end at N; a broken bag is
// reported and pooled as empty (every access stays in [0, N)).
__device__ __forceinline__ void check_bounds(const FwdArgs& a, const Task& k, int32_t nb, int lane, int64_t& start,
                                             int64_t& end) {
  const int32_t g = k.t * a.B + k.b;
  if (start < 0 || end < start || end > a.N || (g == 0 && start != 0) || (g == nb - 1 && end != a.N)) {
    if ((lane & ((1 << k.lsh) - 1)) == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
    start = end = 0;
  }
}

// MINB: resident blocks per SM the register budget targets (R = 8 rows in
// flight per lane needs the registers of two blocks per SM; R = 4 fits three,
// or four with a few values kept in local memory).
template <typename OutT, int R, int DTSEL, bool WT, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) fwd_gather_kernel(const FwdArgs a) {
  __shared__ int32_t s_pref[kMaxSmemTables + 1];
  __shared__ int32_t s_part[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // running task count over tables (block-wide scan, T/256 tables per thread)
  {
    const int per = (a.T + kThreads - 1) / kThreads;
    int32_t mine = 0;
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) {
        const TableMeta m = load_meta(a.meta + t);
        const int G = 32 / lanes_per_row(m, a.lpr_max);
        mine += (a.B + G - 1) / G;
      }
    }
    int32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    int32_t before = 0;
    for (int w = 0; w < warp; ++w) before += s_part[w];
    int32_t run = before + x - mine;
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) {
        s_pref[t] = run;
        const TableMeta m = load_meta(a.meta + t);
        const int G = 32 / lanes_per_row(m, a.lpr_max);
        run += (a.B + G - 1) / G;
      }
    }
    if (tid == kThreads - 1) s_pref[a.T] = run;
    __syncthreads();
  }
  const int32_t ntasks = s_pref[a.T];
  const int32_t nw = (int32_t)((gridDim.x * kThreads) >> 5);
  const int32_t nb = a.T * a.B;
  // the bounds of the warp's next task are requested while this one is pooled
  int32_t task = (int32_t)((blockIdx.x * kThreads + tid) >> 5);
  Task cur = locate_task(a, s_pref, ntasks, task, lane);
  int64_t cs = 0, ce = 0;
  if (cur.live) bag_bounds(a, cur, cs, ce);
  while (task < ntasks) {
    const Task nxt = locate_task(a, s_pref, ntasks, task + nw, lane);
    int64_t ns = 0, ne = 0;
    if (nxt.live) bag_bounds(a, nxt, ns, ne);
    if (cur.live) {
      check_bounds(a, cur, nb, lane, cs, ce);
      const TableMeta m = load_meta(a.meta + cur.t);
      if (DTSEL >= 0) {
        pool_bag_dt<(DTSEL < 0 ? 0 : DTSEL), R, WT, OutT>(a, m, cur.lsh, cur.b, lane, cs, ce);
      } else {
        switch (m.dtype) {
          case TBE_F32: pool_bag_dt<TBE_F32, R, WT, OutT>(a, m, cur.lsh, cur.b, lane, cs, ce); break;
          case TBE_F16: pool_bag_dt<TBE_F16, R, WT, OutT>(a, m, cur.lsh, cur.b, lane, cs, ce); break;
          default: pool_bag_dt<TBE_BF16, R, WT, OutT>(a, m, cur.lsh, cur.b, lane, cs, ce); break;
        }
      }
    }
    cur = nxt;
    cs = ns;
    ce = ne;
    task += nw;
  }
}

// ---------------------------------------------------------------------------
// Ring variant (rows of at most 512 bytes): rows are copied asynchronously
// (cp.async, 16 bytes per lane, cached in L1) into a ring of kRing slots of
// shared memory per lane, so each lane group keeps kRing rows of its bag in
// flight without holding registers for them; lane `sub` copies and later
// reads only its own chunk of each row (no cross-lane ordering needed, the
// per-thread cp.async.wait_group suffices).  The bag's id window sits in
// shared memory, so both the copy of row j + kRing and the sum of row j read
// their id by index.
// ---------------------------------------------------------------------------
constexpr int kRing = 16;      // 16-byte slots per lane
constexpr int kRingStride = kThreads * 16;  // bytes between a thread's ring slots

// KMAX chunks of each row per lane (1, or 2 for rows of 17..32 chunks); the
// ring's kRing slots per lane hold RD = kRing / KMAX rows.
template <int DT, int KMAX, bool WT, typename OutT>
__device__ __forceinline__ void pool_bag_ring(const FwdArgs& a, const TableMeta& m, int lsh, int b, int lane,
                                              int64_t start, int64_t end, uint32_t ring, int32_t* ids, float* wts) {
  constexpr int E = Chunk<DT>::kElems;
  constexpr int RD = kRing / KMAX;  // rows in flight
  const int lpr = 1 << lsh;
  const int C = m.D / E;
  const int sub = lane & (lpr - 1);
  const unsigned vmask = lpr == 32 ? kFull : (((1u << lpr) - 1u) << (lane & ~(lpr - 1)));
  const char* tbl = reinterpret_cast<const char*>(a.weights) + m.w_off;
  const int64_t row_bytes = (int64_t)C * 16;
  const bool weighted = WT && m.weighted;
  const int win = kIdsPerLane * lpr;
  // acc: the running sum, folded into tot every 64 rows so that no serial
  // chain of fp32 adds is longer than 64 + len/64
  float acc[KMAX][E], tot[KMAX][E];
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = tot[k][e] = 0.f;
  int rows_done = 0;
  bool bad = false;
  auto issue = [&](int j, int slot) {  // row j's chunks of this lane into ring slots slot*KMAX + k
    const int32_t id = ids[j];
    if (id >= 0) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int c = sub + k * lpr;
        if (c < C) cp_async16(ring + (slot * KMAX + k) * kRingStride, tbl + (int64_t)id * row_bytes + c * 16);
      }
    }
  };
#pragma unroll 1
  for (int64_t base = start; base < end; base += win) {
    const int nwin = (int)min((int64_t)win, end - base);
#pragma unroll
    for (int k = 0; k < kIdsPerLane; ++k) {  // the window's ids, one coalesced request
      const int idx = k * lpr + sub;
      const uint64_t raw = idx < nwin ? a.indices.id_bits(base + idx) : 0;
      ids[idx] = raw < (uint64_t)m.rows ? (int32_t)raw : -1;
      if (WT) wts[idx] = (weighted && idx < nwin) ? ld_stream_f32(a.psw + base + idx) : 1.f;
    }
    __syncwarp(vmask);
    // rows go in pairs: one copy group, one wait and one loop trip per pair
#pragma unroll 1
    for (int j = 0; j < RD; j += 2) {  // the first RD rows
      if (j < nwin) issue(j, j);
      if (j + 1 < nwin) issue(j + 1, j + 1);
      cp_commit();
    }
#pragma unroll 1
    for (int j = 0; j < nwin; j += 2) {
      cp_wait<RD / 2 - 1>();  // rows j and j + 1 have landed
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jj = j + h;
        if (jj >= nwin) break;
        const int32_t id = ids[jj];
        bad |= id < 0;
        const int slot = jj & (RD - 1);
        const float w = WT ? wts[jj] : 1.f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          const int c = sub + k * lpr;
          float f[E];
          if (c < C && id >= 0) {
            Chunk<DT>::to_float(lds128(ring + (slot * KMAX + k) * kRingStride), f);
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) f[e] = 0.f;
          }
          if (WT && weighted) {
#pragma unroll
            for (int e = 0; e < E; e += 2) mul2(f[e], f[e + 1], w);  // products rounded, then added
          }
#pragma unroll
          for (int e = 0; e < E; e += 2) add2(acc[k][e], acc[k][e + 1], f[e], f[e + 1]);
        }
      }
      if (j + RD < nwin) issue(j + RD, j & (RD - 1));  // refill the two slots just read
      if (j + 1 + RD < nwin) issue(j + 1 + RD, (j + 1) & (RD - 1));
      cp_commit();
      rows_done += 2;
      if ((rows_done & 63) == 0) {
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            add2(tot[k][e], tot[k][e + 1], acc[k][e], acc[k][e + 1]);
            acc[k][e] = acc[k][e + 1] = 0.f;
          }
      }
    }
    __syncwarp(vmask);  // the ids are rewritten by the next window
  }
  OutT* out_row = reinterpret_cast<OutT*>(a.out) + (int64_t)b * a.sumD + m.col_off;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    const int c = sub + k * lpr;
    if (c < C) {
#pragma unroll
      for (int e = 0; e < E; e += 2) add2(acc[k][e], acc[k][e + 1], tot[k][e], tot[k][e + 1]);
      if (a.mean) mean_scale(acc[k], E, end - start);
      store_out<OutT>(out_row + (int64_t)c * E, acc[k], E, a.out_vec_ok);
    }
  }
  if (__any_sync(vmask, bad) && sub == 0) report(a.status, TBE_DEV_BAD_INDEX);
}

template <int DT, bool WT, typename OutT>
__device__ __forceinline__ void pool_ring_dt(const FwdArgs& a, const TableMeta& m, int lsh, int b, int lane,
                                             int64_t start, int64_t end, uint32_t ring, int32_t* ids, float* wts) {
  if (m.D / Chunk<DT>::kElems <= (1 << lsh))
    pool_bag_ring<DT, 1, WT, OutT>(a, m, lsh, b, lane, start, end, ring, ids, wts);
  else
    pool_bag_ring<DT, 2, WT, OutT>(a, m, lsh, b, lane, start, end, ring, ids, wts);
}

// Dynamic shared memory: ring [kRing][kThreads] x 16 B | ids [warps][128] |
// weights [warps][128] | running task count [T + 1].
constexpr size_t kRingBytes = (size_t)kRing * kThreads * 16;
constexpr size_t kRingWinBytes = (size_t)(kThreads / 32) * 128 * 4;

template <typename OutT, int DTSEL, bool WT>
__global__ void __launch_bounds__(kThreads, 3) fwd_ring_kernel(const FwdArgs a) {
  extern __shared__ __align__(16) unsigned char dsm[];
  int32_t* s_ids = reinterpret_cast<int32_t*>(dsm + kRingBytes);
  float* s_wts = reinterpret_cast<float*>(dsm + kRingBytes + kRingWinBytes);
  int32_t* s_pref = reinterpret_cast<int32_t*>(dsm + kRingBytes + 2 * kRingWinBytes);
  __shared__ int32_t s_part[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {  // running task count over tables (as fwd_gather_kernel)
    const int per = (a.T + kThreads - 1) / kThreads;
    int32_t mine = 0;
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) mine += (a.B + (32 / lanes_per_row(load_meta(a.meta + t), a.lpr_max)) - 1) /
                           (32 / lanes_per_row(load_meta(a.meta + t), a.lpr_max));
    }
    int32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    int32_t run = x - mine;
    for (int w = 0; w < warp; ++w) run += s_part[w];
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) {
        s_pref[t] = run;
        const int G = 32 / lanes_per_row(load_meta(a.meta + t), a.lpr_max);
        run += (a.B + G - 1) / G;
      }
    }
    if (tid == kThreads - 1) s_pref[a.T] = run;
    __syncthreads();
  }
  const FwdArgs& ar = a;
  const int32_t ntasks = s_pref[a.T];
  const int32_t nw = (int32_t)((gridDim.x * kThreads) >> 5);
  const int32_t nb = a.T * a.B;
  const uint32_t ring = smem_u32(dsm) + tid * 16;
  int32_t task = (int32_t)((blockIdx.x * kThreads + tid) >> 5);
  Task cur = locate_task(ar, s_pref, ntasks, task, lane);
  int64_t cs = 0, ce = 0;
  if (cur.live) bag_bounds(ar, cur, cs, ce);
  while (task < ntasks) {
    const Task nxt = locate_task(ar, s_pref, ntasks, task + nw, lane);
    int64_t ns = 0, ne = 0;
    if (nxt.live) bag_bounds(ar, nxt, ns, ne);
    if (cur.live) {
      check_bounds(ar, cur, nb, lane, cs, ce);
      const TableMeta m = load_meta(a.meta + cur.t);
      const int vw = lane & ~((1 << cur.lsh) - 1);  // first lane of the virtual warp
      int32_t* ids = s_ids + warp * 128 + vw * kIdsPerLane;
      float* wts = s_wts + warp * 128 + vw * kIdsPerLane;
      if (DTSEL >= 0) {
        pool_ring_dt<(DTSEL < 0 ? 0 : DTSEL), WT, OutT>(ar, m, cur.lsh, cur.b, lane, cs, ce, ring, ids, wts);
      } else {
        switch (m.dtype) {
          case TBE_F32: pool_ring_dt<TBE_F32, WT, OutT>(ar, m, cur.lsh, cur.b, lane, cs, ce, ring, ids, wts); break;
          case TBE_F16: pool_ring_dt<TBE_F16, WT, OutT>(ar, m, cur.lsh, cur.b, lane, cs, ce, ring, ids, wts); break;
          default: pool_ring_dt<TBE_BF16, WT, OutT>(ar, m, cur.lsh, cur.b, lane, cs, ce, ring, ids, wts); break;
        }
      }
    }
    cur = nxt;
    cs = ns;
    ce = ne;
    task += nw;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the block's shared memory
}

template <typename OutT, int DTSEL, bool WT>
int launch_ring(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = kRingBytes + 2 * kRingWinBytes + 4 * ((size_t)a.T + 1);
  auto kern = fwd_ring_kernel<OutT, DTSEL, WT>;
  static size_t configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  if (configured[dev] < smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(96 * 1024 + 4 * (TBE_MAX_TABLES + 1))) !=
        cudaSuccess)
      return TBE_ERR_CUDA;
    configured[dev] = 96 * 1024 + 4 * (TBE_MAX_TABLES + 1);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm <= 0)
    per_sm = 1;
  const int64_t want = ((int64_t)a.T * a.B + (kThreads / 32) - 1) / (kThreads / 32);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * per_sm));
  kern<<<grid, kThreads, smem, s>>>(a);
  return check_launch();
}

template <typename OutT, int DTSEL>
int launch_ring_w(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  if (a.psw != nullptr && p.any_weighted) return launch_ring<OutT, DTSEL, true>(a, s);
  return launch_ring<OutT, DTSEL, false>(a, s);
}

template <typename OutT>
int launch_ring_dt(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  if (p.dtype_mask == (1 << TBE_F16)) return launch_ring_w<OutT, TBE_F16>(p, a, s);
  if (p.dtype_mask == (1 << TBE_F32)) return launch_ring_w<OutT, TBE_F32>(p, a, s);
  if (p.dtype_mask == (1 << TBE_BF16)) return launch_ring_w<OutT, TBE_BF16>(p, a, s);
  return launch_ring_w<OutT, -1>(p, a, s);
}

// ---------------------------------------------------------------------------
// Stream variant (rows of at most 512 bytes; the default).
//
// A warp task is a run of consecutive bags of one table whose length is set
// per table so that every task holds about the same number of lookups (the
// table's mean bag length comes from the offsets at its first and last bag,
// and the target is the batch spread evenly over the grid's warps).  The
// warp reads the bounds of its bags with one request and lays the task's
// lookups out as one stream of positions in shared memory: bag k takes
// plen_k = max(R, len_k rounded up to R) positions, R = 32 / lpr rows per
// step, so the R rows of a step always belong to one bag and every bag (an
// empty one too) ends on a step.  Rows are copied with cp.async into a ring
// of RG groups of four steps per lane and summed group by group (one wait,
// four shared-memory reads, then the adds); the copies run across bag
// boundaries, so the next bags' rows are in flight while a bag is finished.
// Padding positions and ids outside their table are copied with source size
// 0 (the slot is zero-filled and nothing is read), so the summing code has no
// per-row tests.  At the last step of a bag the R row groups' sums are added
// in a fixed butterfly order and group 0 stores the bag.
// ---------------------------------------------------------------------------
constexpr int kSThreads = 128;                       // threads per block
constexpr int kSWarps = kSThreads / 32;
constexpr int kSWin = 256;                           // stream positions staged per warp at once
constexpr int kSGroup = 4;                           // steps per copy group
constexpr int kSWinAlloc = kSWin + kSGroup * 32;     // room for the padding tail of the last group
constexpr int kSRingStride = kSThreads * 16;         // bytes between a thread's ring slots
constexpr int kSTaskMax = 192;                       // most lookups a task is sized for (one window)
constexpr int kFoldGroups = 16;                      // groups (64 steps) summed before acc joins the bag total
constexpr size_t kSSrcBytes = (size_t)kSWarps * kSWinAlloc * 8;
constexpr size_t kSWtsBytes = (size_t)kSWarps * kSWinAlloc * 4;
constexpr size_t kSTotBytes = (size_t)kSThreads * 8 * 4;  // folded sums: 8 floats per thread

// A row of zeros (the widest row the stream kernel takes): padding
// positions and ids outside their table are copied from here.
__device__ __align__(16) unsigned char g_zero_row[512];

// acc[e] += element e of a 16-byte chunk.  Half types use the mixed-precision
// add (fp32 + fp16/bf16 -> fp32, one rounding), which equals converting the
// half exactly to fp32 and adding; fp32 pairs use one packed add.
template <int DT>
__device__ __forceinline__ void accum_chunk(float* acc, const uint4& v) {
  if (DT == TBE_F32) {
    add2(acc[0], acc[1], __uint_as_float(v.x), __uint_as_float(v.y));
    add2(acc[2], acc[3], __uint_as_float(v.z), __uint_as_float(v.w));
  } else {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (DT == TBE_F16)
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
            : "+f"(acc[2 * k]), "+f"(acc[2 * k + 1]) : "r"(w[k]));
      else
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
            : "+f"(acc[2 * k]), "+f"(acc[2 * k + 1]) : "r"(w[k]));
    }
  }
}

struct StreamTask {
  int32_t t, b0, nb;
};

__device__ __forceinline__ StreamTask stream_locate(const int32_t* s_pref, const uint8_t* s_bpt, int32_t T,
                                                    int32_t B, int32_t task) {
  int lo = 0, hi = T - 1;  // table of the task: largest t with s_pref[t] <= task
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= task) lo = mid; else hi = mid - 1;
  }
  StreamTask k;
  k.t = lo;
  const int bpt = s_bpt[lo];
  k.b0 = (task - s_pref[lo]) * bpt;
  k.nb = min(bpt, B - k.b0);
  return k;
}

// Bounds of bag b0 + lane (lanes below nb), requested for a later task.
__device__ __forceinline__ void stream_bounds(const FwdArgs& a, const StreamTask& k, int lane, int64_t& st,
                                              int64_t& en) {
  st = en = 0;
  if (lane < k.nb) {
    const int64_t g = (int64_t)k.t * a.B + k.b0 + lane;
    st = a.offsets.stream(g);
    en = a.offsets.stream(g + 1);
  }
}

// Number of bags of the task whose inclusive padded end is <= p, i.e. the
// bag holding stream position p (p < P).  `pincl` of lanes >= nb is P.
__device__ __forceinline__ int stream_bag_of(int32_t pincl, int32_t p) {
  int k = 0;
#pragma unroll
  for (int step = 16; step > 0; step >>= 1)
    if (__shfl_sync(kFull, pincl, k + step - 1) <= p) k += step;
  return k;
}

// Start of part `part` of a task's padded stream cut into `nparts` parts of
// equal length (multiples of R; part nparts starts at the end, P).
__device__ __forceinline__ int32_t stream_cut(int part, int nparts, int32_t P, int R) {
  if (part >= nparts) return P;
  return (int32_t)(((int64_t)part * P / nparts) & ~(int64_t)(R - 1));
}

// One task: bags b0 .. b0 + nb - 1 of table m; lane k < nb holds the bounds
// [st, en) of bag b0 + k (already checked).  `ring`: this thread's slot 0;
// `srcs` / `wts`: the warp's stream window (row addresses and weights).
// With nparts > 1 every warp of the block pools part `part` (its warp index)
// of the same task: a bag cut by a part boundary is summed in pieces, and
// after a block barrier the part holding its end adds the pieces in part
// order and stores it.
template <int DT, bool WT, typename OutT, int RG, bool MEAN>
__device__ __forceinline__ void stream_task(const FwdArgs& a, const TableMeta& m, const StreamTask& k, int lane,
                                            int32_t st, int32_t en, uint32_t ring, unsigned long long* srcs,
                                            float* wts, float* tot, int part = 0, int nparts = 1) {
  constexpr int E = Chunk<DT>::kElems;
  const int C = m.D / E;  // 16-byte chunks per row (<= 32)
  const int lsh = C <= 1 ? 0 : 32 - __clz(C - 1);
  const int lpr = 1 << lsh, rsh = 5 - lsh, R = 1 << rsh;
  const int grp = lane >> lsh, sub = lane & (lpr - 1);
  const bool live = sub < C;  // lanes past the row's last chunk copy nothing and store nothing
  const bool weighted = WT && m.weighted;
  const char* tbl = reinterpret_cast<const char*>(a.weights) + m.w_off;
  const uint64_t row_bytes = (uint64_t)C * 16u;
  const uint64_t zero_row = reinterpret_cast<uint64_t>(g_zero_row);
  // padded stream: bag k occupies positions [pincl_k - plen_k, pincl_k)
  const int32_t len = lane < k.nb ? en - st : 0;
  const int32_t plen = lane < k.nb ? max(R, (len + R - 1) & ~(R - 1)) : 0;
  int32_t pincl = plen;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(kFull, pincl, o);
    if (lane >= o) pincl += y;
  }
  const int32_t P = __shfl_sync(kFull, pincl, 31);
  const int32_t pst = pincl - plen;
  // this part's positions [lo, hi); its first bag may have begun in an
  // earlier part (head_bag: the piece from lo to its end is kept in the
  // window's spare slots, past any position a window stages) and its last
  // may run on into the next
  const int32_t lo = stream_cut(part, nparts, P, R), hi = stream_cut(part + 1, nparts, P, R);
  int bag = lo < hi && lo > 0 ? stream_bag_of(pincl, lo) : 0;  // bag of the next position pooled
  const int head_bag = nparts > 1 && lo < hi && __shfl_sync(kFull, pst, bag) < lo ? bag : -1;
  bool head_done = false;
  bool bad = false;
  // acc: the running sum since the bag's start or the last fold; tot (this
  // thread's column of shared memory, stride kSThreads): the folded part,
  // valid only while tot_live -- bags longer than kFoldGroups groups
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  bool tot_live = false;
  OutT* out_ptr = reinterpret_cast<OutT*>(a.out) + (int64_t)k.b0 * a.sumD + m.col_off + sub * E;
  const unsigned long long* my_srcs = srcs + grp;
  const float* my_wts = wts + grp;
  const uint32_t sub16 = (uint32_t)sub * 16u;

#pragma unroll 1
  for (int32_t win0 = lo; win0 < hi; win0 += kSWin) {
    const int32_t nwin = min(kSWin, hi - win0);
    const int32_t nsteps = nwin >> rsh;
    const int32_t ngroups = (nsteps + kSGroup - 1) / kSGroup;
    const int32_t npad = (ngroups * kSGroup) << rsh;  // positions of whole groups (<= kSWinAlloc - 31)
    // row addresses (and weights) of positions win0 .. win0 + nwin - 1, then
    // the zero row to npad, 128 positions per round.  The ids (and weights)
    // of every round are copied into the window's slots first and waited for
    // once, so a window waits for one round trip of id loads, not one per
    // round; each slot is then turned into its row's address in place.
    uint32_t valid = 0;  // bit 4 * round + u: slot q0 + 32u + lane holds a lookup
#pragma unroll 1
    for (int32_t q0 = 0, rd = 0; q0 < npad; q0 += 128, ++rd) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int32_t q = q0 + u * 32 + lane;
        const int32_t p = win0 + q;
        const int kb = stream_bag_of(pincl, min(p, P - 1));
        const int32_t r = p - __shfl_sync(kFull, pst, kb);
        const int32_t lk = __shfl_sync(kFull, len, kb);
        const int32_t iu = __shfl_sync(kFull, st, kb) + r;
        if (q0 + u * 32 < npad && q < nwin && r < lk) {
          valid |= 1u << (4 * rd + u);
          a.indices.copy_id(smem_u32(srcs + q), iu);
          if (WT && weighted) cp_async4(smem_u32(wts + q), a.psw + iu);
        }
      }
    }
    cp_commit();
    cp_wait<0>();
#pragma unroll 1
    for (int32_t q0 = 0, rd = 0; q0 < npad; q0 += 128, ++rd) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (q0 + u * 32 < npad) {
          const int32_t q = q0 + u * 32 + lane;
          const bool vu = (valid >> (4 * rd + u)) & 1u;
          const uint64_t raw = vu ? srcs[q] : 0;
          const bool ok = vu && raw < (uint64_t)m.rows;
          bad |= vu && !ok;  // reported; contributes nothing
          srcs[q] = ok ? reinterpret_cast<uint64_t>(tbl) + raw * row_bytes : zero_row;
          if (WT && weighted && !ok) wts[q] = 0.f;
        }
      }
    }
    __syncwarp();
    // steps 4g .. 4g + 3 into the ring slots of group g % RG
    auto issue_group = [&](int32_t g) {
      const uint32_t dst = ring + (uint32_t)((g % RG) * kSGroup) * kSRingStride;
      const unsigned long long* s = my_srcs + ((g * kSGroup) << rsh);
#pragma unroll
      for (int j = 0; j < kSGroup; ++j)
        if (live) cp_async16(dst + j * kSRingStride, reinterpret_cast<const char*>(s[j << rsh] + sub16));
    };
#pragma unroll
    for (int g = 0; g < RG; ++g) {
      if (g < ngroups) issue_group(g);
      cp_commit();
    }
    uint32_t ends = 0;
#pragma unroll 1
    for (int32_t g = 0; g < ngroups; ++g) {
      if ((g & 7) == 0) {  // which of steps 4g .. 4g + 31 end a bag
        const int32_t sj = g * kSGroup + lane;
        const int32_t p = win0 + (sj << rsh);
        const int kb = stream_bag_of(pincl, min(p, P - 1));
        const int32_t kend = __shfl_sync(kFull, pincl, kb);  // every lane takes part in the shuffle
        ends = __ballot_sync(kFull, sj < nsteps && p + R == kend);
      }
      cp_wait<RG - 1>();  // group g has landed
      const uint32_t src = ring + (uint32_t)((g % RG) * kSGroup) * kSRingStride;
      uint4 v[kSGroup];
#pragma unroll
      for (int j = 0; j < kSGroup; ++j) v[j] = lds128(src + j * kSRingStride);
      float w[kSGroup];
      if (WT && weighted) {
#pragma unroll
        for (int j = 0; j < kSGroup; ++j) w[j] = my_wts[(g * kSGroup + j) << rsh];
      }
      const uint32_t eg = ends >> ((g & 7) * kSGroup);
#pragma unroll
      for (int j = 0; j < kSGroup; ++j) {
        if (WT && weighted) {
          float f[E];
          Chunk<DT>::to_float(v[j], f);
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            mul2(f[e], f[e + 1], w[j]);  // the product is rounded to fp32, then added
            add2(acc[e], acc[e + 1], f[e], f[e + 1]);
          }
        } else {
          accum_chunk<DT>(acc, v[j]);
        }
        if (eg & (1u << j)) {  // last step of a bag: combine the row groups and store
          float res[E];
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            res[e] = acc[e];
            res[e + 1] = acc[e + 1];
            if (tot_live) add2(res[e], res[e + 1], tot[e * kSThreads], tot[(e + 1) * kSThreads]);
          }
          for (int o = lpr; o < 32; o <<= 1) {
#pragma unroll
            for (int e = 0; e < E; e += 2)
              add2(res[e], res[e + 1], __shfl_xor_sync(kFull, res[e], o), __shfl_xor_sync(kFull, res[e + 1], o));
          }
          if (nparts > 1 && bag == head_bag) {  // the end of a bag begun in an earlier part: kept for the combine
            if (grp == 0 && live) {
              float* head_piece = reinterpret_cast<float*>(srcs + kSWin + 32) + sub * E;
#pragma unroll
              for (int e = 0; e < E; ++e) head_piece[e] = res[e];
            }
            head_done = true;
          } else {
            if (MEAN) mean_scale(res, E, __shfl_sync(kFull, len, bag));  // lane k holds bag k's length
            if (grp == 0 && live) store_out<OutT>(out_ptr + (int64_t)bag * a.sumD, res, E, a.out_vec_ok);
          }
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = 0.f;
          tot_live = false;
          ++bag;
        }
      }
      if (g + RG < ngroups) issue_group(g + RG);  // refill the slots just read
      cp_commit();
      if ((((win0 >> rsh) / kSGroup + g) & (kFoldGroups - 1)) == kFoldGroups - 1) {  // bound the serial depth of acc
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          float x = acc[e], y = acc[e + 1];
          if (tot_live) add2(x, y, tot[e * kSThreads], tot[(e + 1) * kSThreads]);
          tot[e * kSThreads] = x;
          tot[(e + 1) * kSThreads] = y;
          acc[e] = acc[e + 1] = 0.f;
        }
        tot_live = true;
      }
    }
    __syncwarp();  // the window is rewritten next
  }
  if (__any_sync(kFull, bad) && lane == 0) report(a.status, TBE_DEV_BAD_INDEX);
  if (nparts == 1) return;
  // the last bag runs on into the next part: its piece goes to this thread's
  // ring slots (every copy into them has landed)
  if (lo < hi && hi < P && __shfl_sync(kFull, pincl, stream_bag_of(pincl, hi - 1)) > hi) {
    float res[E];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      res[e] = acc[e];
      res[e + 1] = acc[e + 1];
      if (tot_live) add2(res[e], res[e + 1], tot[e * kSThreads], tot[(e + 1) * kSThreads]);
    }
    for (int o = lpr; o < 32; o <<= 1) {
#pragma unroll
      for (int e = 0; e < E; e += 2)
        add2(res[e], res[e + 1], __shfl_xor_sync(kFull, res[e], o), __shfl_xor_sync(kFull, res[e + 1], o));
    }
    if (grp == 0 && live) {
#pragma unroll
      for (int e = 0; e < E; e += 4)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ring + (uint32_t)(e / 4) * kSRingStride),
                     "f"(res[e]), "f"(res[e + 1]), "f"(res[e + 2]), "f"(res[e + 3])
                     : "memory");
    }
  }
  __syncthreads();  // every part's pieces are in shared memory
  if (head_done) {  // add the pieces of the bag in part order: the parts before this one, then this one's
    const int32_t bstart = __shfl_sync(kFull, pst, head_bag);
    const int32_t hlen = __shfl_sync(kFull, len, head_bag);
    int v0 = part - 1;  // the part holding the bag's first position
    while (v0 > 0 && stream_cut(v0, nparts, P, R) > bstart) --v0;
    if (grp == 0 && live) {
      const float* head_piece = reinterpret_cast<const float*>(srcs + kSWin + 32) + sub * E;
      float res[E];
      bool first = true;
      for (int v = v0; v < part; ++v) {
        if (stream_cut(v, nparts, P, R) == stream_cut(v + 1, nparts, P, R)) continue;  // an empty part
        const uint32_t src = ring - (uint32_t)((part - v) * 32 * 16);  // the same lane of warp v
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const uint4 x = lds128(src + (uint32_t)(e / 4) * kSRingStride);
          const float y[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z), __uint_as_float(x.w)};
          if (first) {
            res[e] = y[0], res[e + 1] = y[1], res[e + 2] = y[2], res[e + 3] = y[3];
          } else {
            add2(res[e], res[e + 1], y[0], y[1]);
            add2(res[e + 2], res[e + 3], y[2], y[3]);
          }
        }
        first = false;
      }
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        if (first) {
          res[e] = head_piece[e], res[e + 1] = head_piece[e + 1];
        } else {
          add2(res[e], res[e + 1], head_piece[e], head_piece[e + 1]);
        }
      }
      if (MEAN) mean_scale(res, E, hlen);
      store_out<OutT>(out_ptr + (int64_t)head_bag * a.sumD, res, E, a.out_vec_ok);
    }
  }
}

// MEAN: mean pooling (a template parameter: the division's code, inlined,
// raised the register pressure of the pooling loop of sum-pooling launches)
template <typename OutT, int DTSEL, bool WT, int RG, int MINB, bool SPLIT, bool MEAN>
__global__ void __launch_bounds__(kSThreads, MINB) fwd_stream_kernel(const FwdArgs a) {
  extern __shared__ __align__(16) unsigned char dsm[];
  constexpr size_t kRingB = (size_t)RG * kSGroup * kSThreads * 16;
  float* s_tot = reinterpret_cast<float*>(dsm + kRingB);
  unsigned long long* s_srcs = reinterpret_cast<unsigned long long*>(dsm + kRingB + kSTotBytes);
  float* s_wts = reinterpret_cast<float*>(dsm + kRingB + kSTotBytes + kSSrcBytes);
  int32_t* s_pref = reinterpret_cast<int32_t*>(dsm + kRingB + kSTotBytes + kSSrcBytes + (WT ? kSWtsBytes : 0));
  uint8_t* s_bpt = reinterpret_cast<uint8_t*>(s_pref + a.T + 1);
  __shared__ int32_t s_part[kSWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t nw = (int32_t)(gridDim.x * kSWarps);
  const int32_t nb_all = a.T * a.B;
  // lookups per task: the batch spread over the grid's warps, 32 .. kSTaskMax
  const int64_t per_task = min((int64_t)kSTaskMax, max((int64_t)32, (a.N + nw - 1) / nw));
  // bags per task at the batch's mean bag length.  Layouts whose tables all
  // have one shape use it for every table, so a task's bags follow from its
  // index alone; other layouts size every table's tasks from its own mean bag
  // length (two offsets per table, read by every block)
  const int bpt_u = a.N > 0 ? (int)min((int64_t)32, max((int64_t)1, (per_task * nb_all + a.N - 1) / a.N)) : 32;
  const int32_t tpt_u = (a.B + bpt_u - 1) / bpt_u;
  int32_t task = (int32_t)blockIdx.x * kSWarps + warp;
  int32_t ntasks = a.T * tpt_u;
  if (a.balance) {  // bags per task and first task of every table (block-wide scan, T/128 tables per thread)
    const int per = (a.T + kSThreads - 1) / kSThreads;
    int32_t mine = 0;
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) {
        const int64_t lo = min(max(a.offsets.ldg((int64_t)t * a.B), (int64_t)0), a.N);
        const int64_t hi = min(max(a.offsets.ldg((int64_t)(t + 1) * a.B), (int64_t)0), a.N);
        const int64_t n = hi - lo;
        const int bpt = n > 0 ? (int)min((int64_t)32, max((int64_t)1, (per_task * a.B + n - 1) / n)) : 32;
        s_bpt[t] = (uint8_t)bpt;
        mine += (a.B + bpt - 1) / bpt;
      }
    }
    int32_t x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    int32_t run = x - mine;
    for (int w = 0; w < warp; ++w) run += s_part[w];
    for (int q = 0; q < per; ++q) {
      const int t = tid * per + q;
      if (t < a.T) {
        s_pref[t] = run;
        run += (a.B + s_bpt[t] - 1) / s_bpt[t];
      }
    }
    if (tid == kSThreads - 1) s_pref[a.T] = run;
    __syncthreads();
    ntasks = s_pref[a.T];
  }
  auto locate = [&](int32_t k) {
    if (a.balance) return stream_locate(s_pref, s_bpt, a.T, a.B, k);
    StreamTask r{k / tpt_u, (k % tpt_u) * bpt_u, 0};
    r.nb = min(bpt_u, a.B - r.b0);
    return r;
  };
  const uint32_t ring = smem_u32(dsm) + tid * 16;
  unsigned long long* srcs = s_srcs + warp * kSWinAlloc;
  float* wts = s_wts + warp * kSWinAlloc;
  if (SPLIT) {  // one task per block, its padded stream cut into one part per warp
    const int32_t nbb = a.split;
    const int32_t tpb = (a.B + nbb - 1) / nbb;
    const int32_t bt = (int32_t)blockIdx.x;
    if (bt < a.T * tpb) {  // the same for the whole block: every warp reaches the combine's barrier
      StreamTask k{bt / tpb, (bt % tpb) * nbb, 0};
      k.nb = min(nbb, a.B - k.b0);
      const TableMeta m = load_meta_now(a.meta + k.t);
      int64_t cs = 0, ce = 0;
      stream_bounds(a, k, lane, cs, ce);
      if (lane < k.nb) {
        const int32_t g = k.t * a.B + k.b0 + lane;
        if (cs < 0 || ce < cs || ce > a.N || (g == 0 && cs != 0) || (g == nb_all - 1 && ce != a.N)) {
          if (warp == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
          cs = ce = 0;
        }
      }
      // split launches take layouts of one table shape, so one dtype
      stream_task<(DTSEL < 0 ? 0 : DTSEL), WT, OutT, RG, MEAN>(a, m, k, lane, (int32_t)cs, (int32_t)ce, ring, srcs, wts,
                                                         s_tot + tid, warp, kSWarps);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }
  StreamTask cur{0, 0, 0};
  int64_t cs = 0, ce = 0;
  if (task < ntasks) {
    cur = locate(task);
    stream_bounds(a, cur, lane, cs, ce);
  }
  while (task < ntasks) {
    // the table's meta is requested before anything waits on the bounds
    const TableMeta m = load_meta_now(a.meta + cur.t);
    // the next task's bounds are requested while this one is pooled
    const int32_t next = task + nw;
    StreamTask nxt{0, 0, 0};
    int64_t ns = 0, ne = 0;
    if (next < ntasks) {
      nxt = locate(next);
      stream_bounds(a, nxt, lane, ns, ne);
    }
    if (lane < cur.nb) {  // offsets must start at 0, never decrease and end at N
      const int32_t g = cur.t * a.B + cur.b0 + lane;
      if (cs < 0 || ce < cs || ce > a.N || (g == 0 && cs != 0) || (g == nb_all - 1 && ce != a.N)) {
        report(a.status, TBE_DEV_BAD_OFFSETS);
        cs = ce = 0;  // pooled as empty
      }
    }
    if (DTSEL >= 0) {
      stream_task<(DTSEL < 0 ? 0 : DTSEL), WT, OutT, RG, MEAN>(a, m, cur, lane, (int32_t)cs, (int32_t)ce, ring, srcs, wts, s_tot + tid);
    } else {
      switch (m.dtype) {
        case TBE_F32: stream_task<TBE_F32, WT, OutT, RG, MEAN>(a, m, cur, lane, (int32_t)cs, (int32_t)ce, ring, srcs, wts, s_tot + tid); break;
        case TBE_F16: stream_task<TBE_F16, WT, OutT, RG, MEAN>(a, m, cur, lane, (int32_t)cs, (int32_t)ce, ring, srcs, wts, s_tot + tid); break;
        default: stream_task<TBE_BF16, WT, OutT, RG, MEAN>(a, m, cur, lane, (int32_t)cs, (int32_t)ce, ring, srcs, wts, s_tot + tid); break;
      }
    }
    cur = nxt;
    cs = ns;
    ce = ne;
    task = next;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the block's shared memory
}

// Split tasks.  The task sizes of the stream kernel are whole bags, so the
// warp that drew the most lookups ends the launch (tasks of 5 Poisson(20)
// bags: 102 positions on average, up to 150).  Where the layout has one
// table shape and a bag per lane covers a block's share of the batch, each
// block instead takes one run of at most 32 bags and its four warps pool
// equal quarters of the run's padded stream (the largest about 118).  The
// piece of a bag that spans two parts is kept in shared memory (at most
// kSplitMaxD fp32 sums in a window's spare slots).
constexpr int kSplitMaxD = (kSWinAlloc - kSWin - 32) * 8 / 4;  // 192
constexpr int64_t kSplitMinPart = 32;                           // positions per part on average, at least

// Bags per block of a split launch of `grid` blocks (0: no split): the
// fewest with which the tables' runs fit in one wave of blocks.
int32_t stream_split_bags(const FwdArgs& a, int grid) {
  if (a.balance || a.N <= 0 || a.T <= 0 || a.B <= 0) return 0;
  int64_t nbb = std::max<int64_t>(1, ((int64_t)a.T * a.B + grid - 1) / grid);
  while (nbb <= 32 && (int64_t)a.T * ((a.B + nbb - 1) / nbb) > grid) ++nbb;
  if (nbb > 32) return 0;
  const int64_t runs = (int64_t)a.T * ((a.B + nbb - 1) / nbb);
  if (a.N < kSplitMinPart * kSWarps * runs) return 0;
  return (int32_t)nbb;
}

constexpr int kStreamRG = 2;    // copy groups in the ring (8 steps in flight per lane)
constexpr int kStreamMinB = 6;  // resident blocks per SM the register budget targets
// The weighted kernel's shared memory (the window's weights too) leaves room
// for 5 blocks per SM, so its register budget targets 5: capped for 6 it
// spilled in the hot loop for no extra residency.
constexpr int kStreamMinBWeighted = 5;

size_t stream_smem_bytes(bool weighted, int32_t T) {
  return (size_t)kStreamRG * kSGroup * kSThreads * 16 + kSTotBytes + kSSrcBytes + (weighted ? kSWtsBytes : 0) +
         5 * ((size_t)T + 1) + 16;
}

template <typename OutT, int DTSEL, bool WT, bool MEAN>
int launch_stream_m(const FwdArgs& a, cudaStream_t s) {
  constexpr int kMinB = WT ? kStreamMinBWeighted : kStreamMinB;
  auto kern = fwd_stream_kernel<OutT, DTSEL, WT, kStreamRG, kMinB, false, MEAN>;
  // split launches need one dtype (a layout of one table shape)
  auto kern_split = fwd_stream_kernel<OutT, DTSEL, WT, kStreamRG, kMinB, (DTSEL >= 0), MEAN>;
  const size_t smem = stream_smem_bytes(WT, a.T);
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  if (!configured[dev]) {
    const int most = (int)stream_smem_bytes(WT, TBE_MAX_TABLES);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, most) != cudaSuccess ||
        cudaFuncSetAttribute(kern_split, cudaFuncAttributeMaxDynamicSharedMemorySize, most) != cudaSuccess)
      return TBE_ERR_CUDA;
    configured[dev] = true;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, smem) != cudaSuccess || per_sm <= 0)
    per_sm = 1;
  if (tuning().fwd_blocks_per_sm > 0) per_sm = std::min(per_sm, tuning().fwd_blocks_per_sm);
  const int64_t want = ((int64_t)a.T * a.B + kSWarps - 1) / kSWarps;  // a bag per warp at least
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * per_sm));
  FwdArgs b = a;
  b.split = a.split && DTSEL >= 0 ? stream_split_bags(a, grid) : 0;
  if (b.split) {
    kern_split<<<grid, kSThreads, smem, s>>>(b);
  } else {
    kern<<<grid, kSThreads, smem, s>>>(b);
  }
  return check_launch();
}

template <typename OutT, int DTSEL, bool WT>
int launch_stream(const FwdArgs& a, cudaStream_t s) {
  return a.mean ? launch_stream_m<OutT, DTSEL, WT, true>(a, s) : launch_stream_m<OutT, DTSEL, WT, false>(a, s);
}

template <typename OutT, int DTSEL>
int launch_stream_w(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  if (a.psw != nullptr && p.any_weighted) return launch_stream<OutT, DTSEL, true>(a, s);
  return launch_stream<OutT, DTSEL, false>(a, s);
}

template <typename OutT>
int launch_stream_dt(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  if (p.dtype_mask == (1 << TBE_F16)) return launch_stream_w<OutT, TBE_F16>(p, a, s);
  if (p.dtype_mask == (1 << TBE_F32)) return launch_stream_w<OutT, TBE_F32>(p, a, s);
  if (p.dtype_mask == (1 << TBE_BF16)) return launch_stream_w<OutT, TBE_BF16>(p, a, s);
  return launch_stream_w<OutT, -1>(p, a, s);
}

bool ring_eligible(const Plan& p) {
  for (int t = 0; t < p.T; ++t)
    if (p.hmeta[t].D * (p.hmeta[t].dtype == TBE_F32 ? 4 : 2) > 512) return false;
  return p.T > 0;
}

template <typename OutT, int R, int DTSEL, bool WT, int MINB>
int launch_typed(const FwdArgs& a, cudaStream_t s) {
  static int occ[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  if (occ[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_gather_kernel<OutT, R, DTSEL, WT, MINB>, kThreads, 0) !=
            cudaSuccess ||
        n <= 0)
      n = 1;
    occ[dev] = n;
  }
  int per_sm = tuning().fwd_blocks_per_sm > 0 ? std::min(tuning().fwd_blocks_per_sm, occ[dev]) : occ[dev];
  const int64_t nb = (int64_t)a.T * a.B;  // upper bound of the warp tasks
  int64_t want = (nb + (kThreads / 32) - 1) / (kThreads / 32);
  int64_t cap = (int64_t)sm_count() * per_sm;
  int grid = (int)std::max<int64_t>(1, std::min(want, cap));
  fwd_gather_kernel<OutT, R, DTSEL, WT, MINB><<<grid, kThreads, 0, s>>>(a);
  return check_launch();
}

template <typename OutT, int DTSEL, bool WT>
int launch_unroll(const FwdArgs& a, cudaStream_t s) {
  if (tuning().fwd_unroll == 8) return launch_typed<OutT, 8, DTSEL, WT, 2>(a, s);
  if (tuning().fwd_blocks_per_sm >= 4) return launch_typed<OutT, 4, DTSEL, WT, 4>(a, s);
  return launch_typed<OutT, 4, DTSEL, WT, 3>(a, s);
}

template <typename OutT, int DTSEL>
int launch_weighted(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  if (a.psw != nullptr && p.any_weighted) return launch_unroll<OutT, DTSEL, true>(a, s);
  return launch_unroll<OutT, DTSEL, false>(a, s);
}

template <typename OutT>
int launch_dtsel(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  // a uniform layout gets a kernel with only that dtype's path
  if (p.dtype_mask == (1 << TBE_F16)) return launch_weighted<OutT, TBE_F16>(p, a, s);
  if (p.dtype_mask == (1 << TBE_F32)) return launch_weighted<OutT, TBE_F32>(p, a, s);
  if (p.dtype_mask == (1 << TBE_BF16)) return launch_weighted<OutT, TBE_BF16>(p, a, s);
  return launch_weighted<OutT, -1>(p, a, s);
}

}  // namespace

// Widest row for which fwd_ring 3 (automatic) takes the stream kernel.  The
// stream kernel keeps 8 steps of R = 512 / row_bytes rows in flight per warp;
// for 512-byte rows (R = 1) that is half of what the per-bag ring keeps, and
// the ring is faster there; for rows up to 256 bytes the stream kernel is
// faster at every batch size measured (2 K .. 33 K lookups per SM).
constexpr int kStreamMaxRowBytes = 256;

// Automatic kernel choice (fwd_ring 3), measured: the stream kernel for rows
// of at most 256 bytes; for rows of up to 512 bytes it still wins on short
// bags (mean under 32 lookups), where it overlaps rows across bags, and the
// per-bag ring, with its deeper queue per bag, wins on long ones.
constexpr int kStreamMaxMeanBag = 32;

int launch_forward_gather(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  const bool short_bags = a.N < (int64_t)kStreamMaxMeanBag * a.T * a.B;
  const int mode = tuning().fwd_ring == 3
                       ? ((p.max_row_bytes <= kStreamMaxRowBytes || (p.max_row_bytes <= 512 && short_bags)) ? 2 : 1)
                       : tuning().fwd_ring;
  if (mode == 2 && ring_eligible(p)) {
    FwdArgs b = a;
    b.split = p.uniform && p.hmeta[0].D <= kSplitMaxD ? 1 : 0;  // a run's bags are chosen at launch
    switch (p.out_dtype) {
      case TBE_F32: return launch_stream_dt<float>(p, b, s);
      case TBE_F16: return launch_stream_dt<__half>(p, b, s);
      default: return launch_stream_dt<__nv_bfloat16>(p, b, s);
    }
  }
  if (mode == 1 && ring_eligible(p)) {
    switch (p.out_dtype) {
      case TBE_F32: return launch_ring_dt<float>(p, a, s);
      case TBE_F16: return launch_ring_dt<__half>(p, a, s);
      default: return launch_ring_dt<__nv_bfloat16>(p, a, s);
    }
  }
  switch (p.out_dtype) {
    case TBE_F32: return launch_dtsel<float>(p, a, s);
    case TBE_F16: return launch_dtsel<__half>(p, a, s);
    default: return launch_dtsel<__nv_bfloat16>(p, a, s);
  }
}

}  // namespace tbe
