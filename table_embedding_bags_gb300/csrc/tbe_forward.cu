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
// lpr = the power of two >= the row's 16-byte chunks (16 lanes for a 256-byte
// fp16 row), so a 32-lane warp pools 32/lpr bags at once without any
// cross-lane reduction.  The VW fetches lpr ids of its bag with one coalesced
// load and hands them around with width-limited shuffles, then requests U
// rows (16-byte loads through the read-only path) before consuming the first,
// keeping U independent index->row chains per lane in flight (the page's
// "several chains" idea, widened to a whole warp).  Warp tasks (32/lpr bags
// of one table) are walked grid-stride by a grid sized to the SM count;
// uniform layouts get a kernel specialised to their one dtype.
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

// Pools one bag with a virtual warp (VW) of `lpr` lanes: every lane owns
// KMAX 16-byte chunks of the row, the VW's lanes fetch `lpr` ids of the bag
// with one coalesced load and hand them around with width-limited
// shuffles, and U rows are requested before the first is consumed.
// KMAX: chunks per lane (1 when the row has <= 32 chunks).
template <int DT, int KMAX, int U, typename OutT>
__device__ __forceinline__ void pool_bag_vw(const FwdArgs& a, const TableMeta& m, int lpr, int32_t g,
                                            int b, int lane) {
  constexpr int E = Chunk<DT>::kElems;           // elements per chunk
  constexpr int NS = (DT == TBE_F32) ? 2 : 1;    // interleaved accumulator sets (fp32 tables)
  const int C = m.D / E;                          // chunks per row
  const int sub = lane & (lpr - 1);
  const unsigned vmask = lpr == 32 ? kFull : (((1u << lpr) - 1u) << (lane & ~(lpr - 1)));
  const char* tbl = reinterpret_cast<const char*>(a.weights) + m.w_off;
  const int64_t row_bytes = (int64_t)C * 16;
  const bool weighted = (a.psw != nullptr) && m.weighted;
  OutT* out_row = reinterpret_cast<OutT*>(a.out) + (int64_t)b * a.sumD + m.col_off;
  const bool vec = a.out_vec_ok;

  // bag bounds: offsets must start at 0, never decrease and end at N; a
  // broken bag is reported and pooled as empty (every access stays in [0, N))
  int64_t o = 0;
  if (sub < 2 && lpr >= 2) o = ld_stream_i64(a.offsets + g + sub);
  int64_t start, end;
  if (lpr >= 2) {
    start = __shfl_sync(vmask, o, 0, lpr);
    end = __shfl_sync(vmask, o, 1, lpr);
  } else {
    start = ld_stream_i64(a.offsets + g);
    end = ld_stream_i64(a.offsets + g + 1);
  }
  const int32_t nb = a.T * a.B;
  if (start < 0 || end < start || end > a.N || (g == 0 && start != 0) || (g == nb - 1 && end != a.N)) {
    if (sub == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
    start = end = 0;
  }

  for (int cb = 0; cb < C; cb += 32 * KMAX) {  // column blocks (rows wider than 32*KMAX chunks)
    float acc[NS][KMAX][E];
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[s][k][e] = 0.f;

    for (int64_t base = start; base < end; base += lpr) {
      const int n = (int)min((int64_t)lpr, end - base);
      int64_t my_id = 0;
      float my_w = 1.f;
      if (sub < n) {
        my_id = ld_stream_i64(a.indices + base + sub);
        if (weighted) my_w = ld_stream_f32(a.psw + base + sub);
      }
      const bool my_ok = (uint64_t)my_id < (uint64_t)m.rows;
      if (__any_sync(vmask, sub < n && !my_ok) && sub == 0 && cb == 0) report(a.status, TBE_DEV_BAD_INDEX);
      for (int j0 = 0; j0 < n; j0 += U) {
        uint4 v[U][KMAX];
        float w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + u;
          const int64_t id = __shfl_sync(vmask, my_id, j, lpr);
          const bool ok = __shfl_sync(vmask, (int)my_ok, j, lpr) && (j < n);
          w[u] = __shfl_sync(vmask, my_w, j, lpr);
          const char* row = tbl + id * row_bytes;
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
#pragma unroll
            for (int e = 0; e < E; ++e) {
              // weighted: the product is rounded to fp32, then added
              const float term = weighted ? __fmul_rn(w[u], f[e]) : f[e];
              acc[u % NS][k][e] = __fadd_rn(acc[u % NS][k][e], term);
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
        store_out<OutT>(out_row + (int64_t)c * E, f, E, vec);
      }
    }
  }
}

template <int DT, int U, typename OutT>
__device__ __forceinline__ void pool_bag_dt(const FwdArgs& a, const TableMeta& m, int lpr, int32_t g, int b,
                                            int lane) {
  constexpr int E = Chunk<DT>::kElems;
  if (m.D / E <= 32)
    pool_bag_vw<DT, 1, U, OutT>(a, m, lpr, g, b, lane);
  else
    pool_bag_vw<DT, 2, (U > 1 ? U / 2 : 1), OutT>(a, m, lpr, g, b, lane);
}

// lanes per row: the power of two >= the row's 16-byte chunks, capped at 32
__device__ __forceinline__ int lanes_per_row(const TableMeta& m) {
  const int C = (m.D * (m.dtype == TBE_F32 ? 4 : 2)) >> 4;
  return C >= 32 ? 32 : (1 << (32 - __clz(C - 1)));
}

constexpr int kMaxSmemTables = TBE_MAX_TABLES;

// Work is enumerated in warp tasks: task k of table t covers bags
// b = k*G_t .. k*G_t + G_t - 1 with G_t = 32 / lanes_per_row (one bag per
// virtual warp).  Every block first builds the running task count of the
// tables in shared memory, then its warps walk the tasks grid-stride.
// DTSEL: the one table dtype of the layout with rows of <= 32 chunks, or -1
// for the generic kernel (any dtype, any width).
template <typename OutT, int U, int DTSEL>
__global__ void __launch_bounds__(kThreads, 3) fwd_gather_kernel(const FwdArgs a) {
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
        const int G = 32 / lanes_per_row(m);
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
        const int G = 32 / lanes_per_row(m);
        run += (a.B + G - 1) / G;
      }
    }
    if (tid == kThreads - 1) s_pref[a.T] = run;
    __syncthreads();
  }
  const int32_t ntasks = s_pref[a.T];
  const int32_t nw = (int32_t)((gridDim.x * kThreads) >> 5);
  for (int32_t task = (int32_t)((blockIdx.x * kThreads + tid) >> 5); task < ntasks; task += nw) {
    int lo = 0, hi = a.T - 1;  // table of this task: largest t with s_pref[t] <= task
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pref[mid] <= task) lo = mid; else hi = mid - 1;
    }
    const int t = lo;
    const TableMeta m = load_meta(a.meta + t);
    const int lpr = lanes_per_row(m);
    const int b = (task - s_pref[t]) * (32 / lpr) + lane / lpr;
    if (b >= a.B) continue;  // the table's last task may have idle virtual warps
    const int32_t g = t * a.B + b;
    if (DTSEL >= 0) {
      pool_bag_vw<(DTSEL < 0 ? 0 : DTSEL), 1, U, OutT>(a, m, lpr, g, b, lane);
    } else {
      switch (m.dtype) {
        case TBE_F32: pool_bag_dt<TBE_F32, U, OutT>(a, m, lpr, g, b, lane); break;
        case TBE_F16: pool_bag_dt<TBE_F16, U, OutT>(a, m, lpr, g, b, lane); break;
        default: pool_bag_dt<TBE_BF16, U, OutT>(a, m, lpr, g, b, lane); break;
      }
    }
  }
}

template <typename OutT, int U, int DTSEL>
int launch_typed(const FwdArgs& a, cudaStream_t s) {
  static int occ[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  if (occ[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_gather_kernel<OutT, U, DTSEL>, kThreads, 0) !=
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
  fwd_gather_kernel<OutT, U, DTSEL><<<grid, kThreads, 0, s>>>(a);
  return check_launch();
}

template <typename OutT, int DTSEL>
int launch_unroll(const FwdArgs& a, cudaStream_t s) {
  switch (tuning().fwd_unroll) {
    case 2:
    case 4: return launch_typed<OutT, 4, DTSEL>(a, s);
    default: return launch_typed<OutT, 8, DTSEL>(a, s);
  }
}

template <typename OutT>
int launch_dtsel(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  // a uniform layout whose rows fit one chunk per lane gets a kernel with
  // only that dtype's path (fewer live registers, more resident warps)
  bool narrow = true;
  for (int t = 0; t < p.T; ++t)
    if (p.hmeta[t].D * (p.hmeta[t].dtype == TBE_F32 ? 4 : 2) > 512) narrow = false;
  if (narrow && p.dtype_mask == (1 << TBE_F16)) return launch_unroll<OutT, TBE_F16>(a, s);
  if (narrow && p.dtype_mask == (1 << TBE_F32)) return launch_unroll<OutT, TBE_F32>(a, s);
  if (narrow && p.dtype_mask == (1 << TBE_BF16)) return launch_unroll<OutT, TBE_BF16>(a, s);
  return launch_unroll<OutT, -1>(a, s);
}

}  // namespace

int launch_forward_gather(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  switch (p.out_dtype) {
    case TBE_F32: return launch_dtsel<float>(p, a, s);
    case TBE_F16: return launch_dtsel<__half>(p, a, s);
    default: return launch_dtsel<__nv_bfloat16>(p, a, s);
  }
}

}  // namespace tbe
