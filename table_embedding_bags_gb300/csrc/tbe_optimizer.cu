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
// per-table unique counts.  One warp owns one distinct row at a time (rows
// are distinct, so no two warps touch the same weights or momentum), lanes
// cover the row four columns each; Adagrad sums the squares with a warp
// reduction, then every lane applies w - step * g as one fused multiply-add
// and stores it rounded to nearest-even in the table's dtype.
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

// Four consecutive elements of a table row, as floats and back (stores round
// to nearest-even).  Callers keep the address 8-byte aligned (16 for fp32):
// rows start on 16-byte boundaries and the column is a multiple of 4.
template <int DT>
struct Quad;

template <>
struct Quad<TBE_F32> {
  static constexpr int kBytes = 16;
  __device__ __forceinline__ static float4 load(const uint8_t* p) { return *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ static void store(uint8_t* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};

template <>
struct Quad<TBE_F16> {
  static constexpr int kBytes = 8;
  __device__ __forceinline__ static float4 load(const uint8_t* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ __forceinline__ static void store(uint8_t* p, float4 v) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

template <>
struct Quad<TBE_BF16> {
  static constexpr int kBytes = 8;
  __device__ __forceinline__ static float4 load(const uint8_t* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);  // bf16 -> fp32 is exact: the bits move up
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  }
  __device__ __forceinline__ static void store(uint8_t* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

// w <- w - step * g over one row, lanes striding by 32 quads.
template <int DT>
__device__ __forceinline__ void apply_row(uint8_t* wrow, const float* g, int D, float step, int lane) {
  for (int c = lane * 4; c < D; c += 128) {
    const float4 gv = *reinterpret_cast<const float4*>(g + c);
    uint8_t* p = wrow + (size_t)c * (Quad<DT>::kBytes / 4);
    float4 w = Quad<DT>::load(p);
    w.x = fmaf(-step, gv.x, w.x);
    w.y = fmaf(-step, gv.y, w.y);
    w.z = fmaf(-step, gv.z, w.z);
    w.w = fmaf(-step, gv.w, w.w);
    Quad<DT>::store(p, w);
  }
}

template <int KIND>
__global__ void __launch_bounds__(kUpdThreads) exact_update_kernel(UpdArgs a) {
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
  const int64_t stride = (int64_t)gridDim.x * kUpdWarps;
  for (int64_t u = (int64_t)blockIdx.x * kUpdWarps + warp; u < U; u += stride) {
    int lo = 0, hi = a.T - 1;  // the table of run u: the last t with s_uc[t] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_uc[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    const TableMeta m = a.meta[lo];
    const int64_t row = a.unique_rows[u];
    const int64_t id = row - m.row_base;
    const int64_t go = s_go[lo] + (u - s_uc[lo]) * (int64_t)m.D;
    if (id < 0 || id >= m.rows) {
      if (lane == 0) report(a.status, TBE_DEV_BAD_INDEX);
      continue;
    }
    if (go < 0 || go + m.D > a.row_grads_capacity) {
      if (lane == 0) report(a.status, TBE_DEV_CAPACITY);
      continue;
    }
    const float* g = a.row_grads + go;
    float step = a.lr;
    if (KIND == TBE_OPT_EXACT_ROWWISE_ADAGRAD) {
      float ss = 0.f;
      for (int c = lane * 4; c < m.D; c += 128) {
        const float4 v = *reinterpret_cast<const float4*>(g + c);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
      const float m_new = __fadd_rn(a.momentum[row], __fdiv_rn(ss, (float)m.D));
      __syncwarp();  // every lane has read the old value before lane 0 replaces it
      if (lane == 0) a.momentum[row] = m_new;
      step = __fdiv_rn(a.lr, __fadd_rn(__fsqrt_rn(m_new), a.eps));
    }
    uint8_t* wrow = a.weights + m.w_off + id * (int64_t)m.D * (m.dtype == TBE_F32 ? 4 : 2);
    if (m.dtype == TBE_F32) apply_row<TBE_F32>(wrow, g, m.D, step, lane);
    else if (m.dtype == TBE_F16) apply_row<TBE_F16>(wrow, g, m.D, step, lane);
    else apply_row<TBE_BF16>(wrow, g, m.D, step, lane);
  }
}

template <int KIND>
int launch_kind(const UpdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(int64_t) * 2 * (size_t)(a.T + 1);
  auto kernel = exact_update_kernel<KIND>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TBE_ERR_CUDA;
  int64_t want = (a.max_unique + kUpdWarps - 1) / kUpdWarps;
  const int64_t cap = 4LL * sm_count();
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
