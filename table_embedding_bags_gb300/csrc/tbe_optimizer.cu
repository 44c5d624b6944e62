// tbe_optimizer.cu -- exact optimizer step on the backward's row gradients.
//
// [FBT] "Why the backward is the hard half": TBE never hands the table-sized
// gradient to a separate optimizer; each distinct row is updated once, from
// its finished gradient g (the sum over the row's run), which is what makes
// a nonlinear update such as row-wise Adagrad "exact".  Two kinds:
//   exact SGD:              W[r] <- W[r] - lr * g
//   exact row-wise Adagrad: m[r] <- m[r] + (sum_c g_c^2) / D_t
//                           W[r] <- W[r] - lr / (sqrt(m[r]) + eps) * g
// (one FP32 momentum scalar per global row).
//
// This kernel runs after the backward on the same stream and reads its
// outputs as they are: unique_rows, the table-major row_grads blocks and the
// per-table unique counts.  A warp owns a group of consecutive distinct rows
// at a time (rows are distinct, so no two warps touch the same weights or
// momentum) and lanes cover a row four columns each; Adagrad sums the
// squares with a warp reduction, then every lane applies w - step * g as one
// fused multiply-add and stores it rounded to nearest-even in the table's
// dtype.
//
// Per block, the per-table counts and the start of each table's gradient
// block (sum over earlier tables of rows * D) are staged in shared memory.
// The kernel is launched with programmatic stream serialisation, so its
// launch overlaps the end of the backward's last kernel; it reads nothing
// before griddepcontrol.wait.
#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kUpdThreads = 256;
constexpr int kUpdWarps = kUpdThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void wait_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Where one distinct row's update reads and writes.
struct RowJob {
  const float* g;   // its gradient (D floats)
  uint8_t* w;       // its weights
  int64_t row;      // global row (momentum index)
  int32_t D;
  int32_t dtype;
  bool ok;
};

// Rows per warp in flight: a warp updates kRowsPerWarp rows of its tile at
// once, loading the gradient, weights and momentum of all of them before it
// computes any (a row of up to 128 columns is one quad per lane), so one
// memory latency is spent per group instead of one per row.  Wider rows go
// through a column loop afterwards.
constexpr int kRowsPerWarp = 4;

template <int KIND>
__device__ __forceinline__ float row_step(const UpdArgs& a, float m_old, float ss, int D, float* m_new) {
  if (KIND != TBE_OPT_EXACT_ROWWISE_ADAGRAD) return a.lr;
  return adagrad_step(a.lr, a.eps, m_old, ss, D, m_new);
}

template <int KIND>
__global__ void __launch_bounds__(kUpdThreads, 3) exact_update_kernel(UpdArgs a) {
  extern __shared__ int64_t s_upd[];
  int64_t* s_uc = s_upd;             // [T+1] distinct rows of tables < t
  int64_t* s_go = s_upd + a.T + 1;   // [T+1] float offset of table t's gradient block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  wait_predecessor();
  for (int i = threadIdx.x; i <= a.T; i += kUpdThreads) s_uc[i] = a.unique_count[i];
  __syncthreads();
  if (warp == 0) {  // exclusive running sum of (rows of t) * D_t, 32 tables per round
    int64_t run = 0;
    for (int base = 0; base < a.T; base += 32) {
      const int t = base + lane;
      const int64_t own = t < a.T ? (s_uc[t + 1] - s_uc[t]) * (int64_t)a.meta[t].D : 0;
      int64_t inc = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += n;
      }
      if (t < a.T) s_go[t] = run + inc - own;
      run += __shfl_sync(kFull, inc, 31);
    }
    if (lane == 0) s_go[a.T] = run;
  }
  __syncthreads();

  int64_t U = s_uc[a.T];
  if (U > a.max_unique) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, TBE_DEV_CAPACITY);
    U = a.max_unique;
  }
  // A warp takes a tile of 32 consecutive runs: lane l looks up run t0 + l
  // (its row id, table, gradient offset and weight row) in one coalesced
  // pass and leaves the result in the warp's shared-memory slots, then the
  // warp updates the tile's rows kRowsPerWarp at a time.
  __shared__ int64_t s_row[kUpdWarps][32], s_gofs[kUpdWarps][32], s_wofs[kUpdWarps][32];
  __shared__ int32_t s_D[kUpdWarps][32], s_kind[kUpdWarps][32];  // width; dtype | ok << 8
  const int64_t stride = (int64_t)gridDim.x * kUpdWarps * 32;
  for (int64_t t0 = ((int64_t)blockIdx.x * kUpdWarps + warp) * 32; t0 < U; t0 += stride) {
    const int64_t u_me = t0 + lane;
    bool ok_me = false;
    int64_t row_me = 0, go_me = 0, wo_me = 0;
    int32_t D_me = 0, dt_me = TBE_F32;
    if (u_me < U) {
      row_me = a.unique_rows[u_me];
      int lo = 0, hi = a.T - 1;  // the table of run u: the last t with s_uc[t] <= u
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_uc[mid] <= u_me) lo = mid;
        else hi = mid - 1;
      }
      const TableMeta m = a.meta[lo];
      const int64_t id = row_me - m.row_base;
      go_me = s_go[lo] + (u_me - s_uc[lo]) * (int64_t)m.D;
      if (id < 0 || id >= m.rows) {
        report(a.status, TBE_DEV_BAD_INDEX);
      } else if (go_me < 0 || go_me + m.D > a.row_grads_capacity) {
        report(a.status, TBE_DEV_CAPACITY);
      } else {
        ok_me = true;
        D_me = m.D;
        dt_me = m.dtype;
        wo_me = m.w_off + id * (int64_t)m.D * (m.dtype == TBE_F32 ? 4 : 2);
      }
    }
    s_row[warp][lane] = row_me;
    s_gofs[warp][lane] = go_me;
    s_wofs[warp][lane] = wo_me;
    s_D[warp][lane] = D_me;
    s_kind[warp][lane] = dt_me | ((int)ok_me << 8);
    __syncwarp();
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += kRowsPerWarp) {
      if (t0 + r0 >= U) break;
      RowJob job[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int src = r0 + r;
        const int32_t kind = s_kind[warp][src];
        job[r].ok = (kind >> 8) != 0;
        job[r].D = s_D[warp][src];
        job[r].dtype = kind & 0xff;
        job[r].row = s_row[warp][src];
        job[r].g = job[r].ok ? a.row_grads + s_gofs[warp][src] : nullptr;
        job[r].w = job[r].ok ? a.weights + s_wofs[warp][src] : nullptr;
      }
      // rows of at most 128 columns: every load of the group first, then the math
      float4 gv[kRowsPerWarp], wv[kRowsPerWarp];
      float mo[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        gv[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        wv[r] = gv[r];
        mo[r] = 0.f;
        const bool narrow = job[r].ok && job[r].D <= 128;
        if (narrow && lane * 4 < job[r].D) {
          gv[r] = *reinterpret_cast<const float4*>(job[r].g + lane * 4);
          wv[r] = load_quad(job[r].dtype, job[r].w + (size_t)lane * (job[r].dtype == TBE_F32 ? 16 : 8));
        }
        if (KIND == TBE_OPT_EXACT_ROWWISE_ADAGRAD && narrow) mo[r] = a.momentum[job[r].row];
      }
      float ss[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) ss[r] = sum_sq(gv[r], 0.f);
      if (KIND == TBE_OPT_EXACT_ROWWISE_ADAGRAD) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) ss[r] = warp_sum(ss[r]);
      }
      __syncwarp();  // every lane has read the old momentum before it is replaced
      // lane r < kRowsPerWarp works out row r's momentum and step (one square
      // root and two divides per lane instead of per row), then hands the step
      // round; rows wider than 128 columns are done below
      float step[kRowsPerWarp];
      if (KIND == TBE_OPT_EXACT_ROWWISE_ADAGRAD) {
        float m_sel = 0.f, ss_sel = 0.f;
        int D_sel = 1;
        bool mine = false;
        int64_t row_sel = 0;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
          if (lane == r) {
            m_sel = mo[r];
            ss_sel = ss[r];
            D_sel = job[r].D > 0 ? job[r].D : 1;
            mine = job[r].ok && job[r].D <= 128;
            row_sel = job[r].row;
          }
        float m_new = 0.f;
        const float st = row_step<KIND>(a, m_sel, ss_sel, D_sel, &m_new);
        if (mine) a.momentum[row_sel] = m_new;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) step[r] = __shfl_sync(kFull, st, r);
      } else {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) step[r] = a.lr;
      }
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        if (!job[r].ok || job[r].D > 128) continue;
        if (lane * 4 < job[r].D)
          store_quad(job[r].dtype, job[r].w + (size_t)lane * (job[r].dtype == TBE_F32 ? 16 : 8),
                     fma_quad(step[r], gv[r], wv[r]));
      }
      // wider rows: a column loop per row (two passes over the gradient for Adagrad)
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        if (!job[r].ok || job[r].D <= 128) continue;
        const int D = job[r].D, dt = job[r].dtype, eb = dt == TBE_F32 ? 4 : 2;
        float step = a.lr;
        if (KIND == TBE_OPT_EXACT_ROWWISE_ADAGRAD) {
          float acc = 0.f;
          for (int c = lane * 4; c < D; c += 128) acc = sum_sq(*reinterpret_cast<const float4*>(job[r].g + c), acc);
          acc = warp_sum(acc);
          const float m_old = a.momentum[job[r].row];
          __syncwarp();
          float m_new = 0.f;
          step = row_step<KIND>(a, m_old, acc, D, &m_new);
          if (lane == 0) a.momentum[job[r].row] = m_new;
        }
        for (int c = lane * 4; c < D; c += 128) {
          uint8_t* p = job[r].w + (size_t)c * eb;
          store_quad(dt, p, fma_quad(step, *reinterpret_cast<const float4*>(job[r].g + c), load_quad(dt, p)));
        }
      }
    }
    __syncwarp();  // the tile's slots are rewritten by the next tile
  }
}

template <int KIND>
int launch_kind(const UpdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(int64_t) * 2 * (size_t)(a.T + 1);
  auto kernel = exact_update_kernel<KIND>;
  if (smem > 32 * 1024 &&  // beyond the default once the kernel's static slots are counted
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TBE_ERR_CUDA;
  // a grid-stride loop over tiles of 32 runs per warp: at most as many
  // blocks as fit on the GPU at once, fewer for small batches
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kUpdThreads, smem) != cudaSuccess ||
      per_sm <= 0)
    per_sm = 1;
  const int64_t want = (a.max_unique + kUpdWarps * 32 - 1) / (kUpdWarps * 32);
  const int64_t cap = (int64_t)per_sm * sm_count();
  const int grid = (int)(want < 1 ? 1 : (want > cap ? cap : want));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)kUpdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, a) != cudaSuccess) return TBE_ERR_CUDA;
  return check_launch();
}

}  // namespace

int launch_exact_update(const Plan& p, const UpdArgs& a, cudaStream_t s) {
  (void)p;
  if (a.max_unique == 0) return TBE_OK;
  const int st = a.kind == TBE_OPT_EXACT_ROWWISE_ADAGRAD ? launch_kind<TBE_OPT_EXACT_ROWWISE_ADAGRAD>(a, s)
                                                          : launch_kind<TBE_OPT_EXACT_SGD>(a, s);
  trace_mark(s, "exact_update");
  return st;
}

}  // namespace tbe
