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
    const int64_t raw = idx < nwin ? ld_stream_i64(a.indices + base + idx) : 0;
    iw.id[k] = (uint64_t)raw < (uint64_t)m.rows ? (int32_t)raw : -1;
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
  start = ld_stream_i64(a.offsets + g);
  end = ld_stream_i64(a.offsets + g + 1);
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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the N most recent groups of this thread have landed
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

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
  float acc[KMAX][E];  // one accumulator set: rows arrive far slower than adds complete
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[k][e] = 0.f;
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
      const int64_t raw = idx < nwin ? ld_stream_i64(a.indices + base + idx) : 0;
      ids[idx] = (uint64_t)raw < (uint64_t)m.rows ? (int32_t)raw : -1;
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
    }
    __syncwarp(vmask);  // the ids are rewritten by the next window
  }
  OutT* out_row = reinterpret_cast<OutT*>(a.out) + (int64_t)b * a.sumD + m.col_off;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    const int c = sub + k * lpr;
    if (c < C) {
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

int launch_forward_gather(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  if (tuning().fwd_ring && ring_eligible(p)) {
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
