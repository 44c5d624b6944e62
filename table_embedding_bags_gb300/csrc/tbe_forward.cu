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
// Design (GB300): a grid sized to the SM count whose warps walk bags
// g = t*B + b in a grid-stride loop, one bag per warp at a time.  A row of
// D_t elements is split into 16-byte chunks; `lpr` lanes (a power of two)
// cover one row and the warp's 32/lpr lane groups take different lookups of
// the same bag, so a bag keeps (32/lpr) * U independent index->row chains in
// flight (the page's "several chains" idea, widened to a full warp).  The
// bag's ids and weights are fetched 32 at a time with one coalesced load and
// handed to the lane groups by shuffles, which breaks the index->row
// dependency chain for all but the first 32 ids.  Partial sums of the lane
// groups are combined with xor-shuffles at the end of the bag.
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

// Pools bag (t, b) = positions [start, end) of a table of element type DT.
// KMAX: 16-byte chunks per lane per row (1 when the row has <= 32 chunks).
// U: lookups per lane group issued before their rows are consumed.
template <int DT, int KMAX, int U, typename OutT>
__device__ __forceinline__ void pool_bag(const FwdArgs& a, const TableMeta& m, int64_t start,
                                         int64_t end, int b, int lane) {
  constexpr int E = Chunk<DT>::kElems;           // elements per chunk
  constexpr int NS = (DT == TBE_F32) ? 2 : 1;    // interleaved accumulator sets (fp32 tables)
  const int C = m.D / E;                          // chunks per row
  const int lpr = C >= 32 ? 32 : (1 << (32 - __clz(C - 1)));
  const int G = 32 / lpr;
  const int grp = lane / lpr;
  const int sub = lane & (lpr - 1);
  const char* tbl = reinterpret_cast<const char*>(a.weights) + m.w_off;
  const int64_t row_bytes = (int64_t)C * 16;
  const bool weighted = (a.psw != nullptr) && m.weighted;
  OutT* out_row = reinterpret_cast<OutT*>(a.out) + (int64_t)b * a.sumD + m.col_off;
  const bool vec = a.out_vec_ok;

  for (int cb = 0; cb < C; cb += 32 * KMAX) {  // column blocks (rows wider than 32*KMAX chunks)
    float acc[NS][KMAX][E];
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[s][k][e] = 0.f;

    for (int64_t base = start; base < end; base += 32) {
      const int n = (int)min((int64_t)32, end - base);
      int64_t my_id = 0;
      float my_w = 1.f;
      if (lane < n) {
        my_id = ld_stream_i64(a.indices + base + lane);
        if (weighted) my_w = ld_stream_f32(a.psw + base + lane);
      }
      const bool my_ok = (uint64_t)my_id < (uint64_t)m.rows;
      if (__any_sync(kFull, lane < n && !my_ok) && lane == 0 && cb == 0)
        report(a.status, TBE_DEV_BAD_INDEX);

      for (int j0 = 0; j0 < n; j0 += G * U) {
        uint4 v[U][KMAX];
        float w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = j0 + u * G + grp;
          const int src = j & 31;
          const int64_t id = __shfl_sync(kFull, my_id, src);
          const bool ok = __shfl_sync(kFull, (int)my_ok, src) && (j < n);
          w[u] = __shfl_sync(kFull, my_w, src);
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
    // combine accumulator sets, then the lane groups
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        float x = acc[0][k][e];
        if (NS == 2) x = __fadd_rn(x, acc[NS - 1][k][e]);
        for (int off = lpr; off < 32; off <<= 1) x = __fadd_rn(x, __shfl_xor_sync(kFull, x, off));
        acc[0][k][e] = x;
      }
    if (grp == 0) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int c = cb + sub + k * lpr;
        if (c < C) store_out<OutT>(out_row + (int64_t)c * E, acc[0][k], E, vec);
      }
    }
  }
}

template <int DT, int U, typename OutT>
__device__ __forceinline__ void pool_bag_dt(const FwdArgs& a, const TableMeta& m, int64_t start,
                                            int64_t end, int b, int lane) {
  constexpr int E = Chunk<DT>::kElems;
  if (m.D / E <= 32)
    pool_bag<DT, 1, U, OutT>(a, m, start, end, b, lane);
  else
    pool_bag<DT, 2, (U > 1 ? U / 2 : 1), OutT>(a, m, start, end, b, lane);
}

template <typename OutT, int U>
__global__ void __launch_bounds__(kThreads) fwd_gather_kernel(const FwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int32_t nb = a.T * a.B;
  const int32_t nw = (int32_t)((gridDim.x * kThreads) >> 5);
  for (int32_t g = (int32_t)((blockIdx.x * kThreads + threadIdx.x) >> 5); g < nb; g += nw) {
    const int t = g / a.B;
    const int b = g - t * a.B;
    int64_t o = 0;
    if (lane < 2) o = ld_stream_i64(a.offsets + g + lane);
    int64_t start = __shfl_sync(kFull, o, 0);
    int64_t end = __shfl_sync(kFull, o, 1);
    // offsets must start at 0, never decrease and end at N; a broken bag is
    // reported and pooled as empty (every access stays inside [0, N))
    bool bad = start < 0 || end < start || end > a.N || (g == 0 && start != 0) ||
               (g == nb - 1 && end != a.N);
    if (bad) {
      if (lane == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
      start = end = 0;
    }
    const TableMeta m = load_meta(a.meta + t);
    switch (m.dtype) {
      case TBE_F32: pool_bag_dt<TBE_F32, U, OutT>(a, m, start, end, b, lane); break;
      case TBE_F16: pool_bag_dt<TBE_F16, U, OutT>(a, m, start, end, b, lane); break;
      default: pool_bag_dt<TBE_BF16, U, OutT>(a, m, start, end, b, lane); break;
    }
  }
}

template <typename OutT, int U>
int launch_typed(const FwdArgs& a, cudaStream_t s) {
  static int occ[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) dev = 63;
  if (occ[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_gather_kernel<OutT, U>, kThreads, 0) !=
        cudaSuccess || n <= 0)
      n = 1;
    occ[dev] = n;
  }
  int per_sm = tuning().fwd_blocks_per_sm > 0 ? std::min(tuning().fwd_blocks_per_sm, occ[dev]) : occ[dev];
  const int64_t nb = (int64_t)a.T * a.B;
  int64_t want = (nb + (kThreads / 32) - 1) / (kThreads / 32);
  int64_t cap = (int64_t)sm_count() * per_sm;
  int grid = (int)std::max<int64_t>(1, std::min(want, cap));
  fwd_gather_kernel<OutT, U><<<grid, kThreads, 0, s>>>(a);
  return check_launch();
}

template <typename OutT>
int launch_unroll(const FwdArgs& a, cudaStream_t s) {
  switch (tuning().fwd_unroll) {
    case 2: return launch_typed<OutT, 2>(a, s);
    case 4: return launch_typed<OutT, 4>(a, s);
    default: return launch_typed<OutT, 8>(a, s);
  }
}

}  // namespace

int launch_forward_gather(const Plan& p, const FwdArgs& a, cudaStream_t s) {
  switch (p.out_dtype) {
    case TBE_F32: return launch_unroll<float>(a, s);
    case TBE_F16: return launch_unroll<__half>(a, s);
    default: return launch_unroll<__nv_bfloat16>(a, s);
  }
}

}  // namespace tbe
