// tbe_internal.cuh -- shared definitions of the libtbe translation units.
//
// Page cited throughout: "FBTriton table-batched embeddings: the backward win
// is a threshold moved from 32 to 256" ([FBT] + section title).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tbe.h"

namespace tbe {

// Packed per-table metadata, one 32-byte record per table plus a sentinel
// record T whose row_base is the total row count.  Lives in device memory
// owned by the caller (see tbe_plan_create) and is read through the
// read-only cache; every warp reads the record of the table it works on.
struct __align__(16) TableMeta {
  int64_t w_off;     // byte offset of the table in the packed weight buffer
  int64_t row_base;  // global row of id 0 ([FBT] hash_size_cumsum[t])
  int32_t rows;      // rows of the table
  int32_t col_off;   // output column offset (D_offsets[t])
  int32_t D;         // width
  uint8_t dtype;     // TBE_F32 / TBE_F16 / TBE_BF16
  uint8_t weighted;  // lookups of this table are scaled by per-sample weights
  uint8_t pad[2];
};
static_assert(sizeof(TableMeta) == 32, "TableMeta must stay 32 bytes");

// Host-side plan.
struct Plan {
  int32_t T;
  int32_t out_dtype;
  int32_t sumD;
  int32_t maxD;
  int64_t total_rows;
  int32_t key_bits;      // bits needed for a global row or the sentinel total_rows
  int32_t seg_bits;      // bits needed for an id or the value rows_t, over all tables
  int32_t dtype_mask;    // bit d set if some table has dtype d
  int32_t any_weighted;  // some table is marked weighted
  int32_t out_vec_ok;    // every output segment start is 16-byte aligned
  int32_t uniform;       // every table has the same width, dtype and weighting
  int32_t max_row_bytes; // widest row of the layout
  int32_t hist_ok;       // static part of the histogram-path eligibility
  int32_t pooling;       // TBE_POOL_SUM or TBE_POOL_MEAN
  int32_t device;        // device the plan was created on
  const TableMeta* dmeta;  // device copy (caller memory)
  TableMeta* hmeta;        // host copy (T+1 records)
};

// Process-wide tuning (tbe_set_tuning).
struct Tuning {
  int32_t long_run_threshold;
  int32_t long_chunk;
  int32_t fwd_unroll;
  int32_t fwd_blocks_per_sm;
  int32_t hist_min_mean_bag;
  int32_t short_item_lookups;
  int32_t fwd_lanes_per_row;
  int32_t red_unroll;
  int32_t fwd_ring;
};
const Tuning& tuning();

// Stage tracing (tbe_trace_enable / tbe_trace_read).
void trace_begin(cudaStream_t s);
void trace_mark(cudaStream_t s, const char* name);

int sm_count();
int check_launch();  // TBE_OK or TBE_ERR_CUDA after a kernel launch

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

// 16-byte read-only load of table rows (several rows of one bag are in
// flight at once; the read-only path keeps hot rows in L1/L2).
__device__ __forceinline__ uint4 ld_row16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Streaming 8-byte load for index / offset arrays that are read once.
__device__ __forceinline__ int64_t ld_stream_i64(const int64_t* p) {
  int64_t v;
  asm volatile("ld.global.nc.L1::no_allocate.s64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// An index or offset array: int64 (the default entry points) or int32 (the
// *_i32 entry points).  The flag is the same for a whole launch.
struct IdxPtr {
  const void* p;
  int32_t i32;
  // read once, not kept in L1
  __device__ __forceinline__ int64_t stream(int64_t i) const {
    if (i32) {
      int32_t v;
      asm volatile("ld.global.nc.L1::no_allocate.s32 %0, [%1];" : "=r"(v) : "l"(static_cast<const int32_t*>(p) + i));
      return v;
    }
    int64_t v;
    asm volatile("ld.global.nc.L1::no_allocate.s64 %0, [%1];" : "=l"(v) : "l"(static_cast<const int64_t*>(p) + i));
    return v;
  }
  // A row id as raw bits, read once: int64 ids as stored, int32 ids
  // zero-extended by the load itself.  A negative int32 id then reads as a
  // value of at least 2^31, out of range for every table exactly like its
  // int64 form, so callers compare it (unsigned) with a row count and use
  // only in-range values; nothing has to wait for the load to extend it.
  __device__ __forceinline__ uint64_t id_bits(int64_t i) const {
    uint64_t v;
    if (i32)
      asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=l"(v) : "l"(static_cast<const int32_t*>(p) + i));
    else
      asm volatile("ld.global.nc.L1::no_allocate.u64 %0, [%1];" : "=l"(v) : "l"(static_cast<const int64_t*>(p) + i));
    return v;
  }
  // Id i copied into the 8-byte shared-memory slot at dst (asynchronously,
  // cp.async): int64 ids as stored, int32 ids into the low word with the
  // high word zeroed, so the slot reads as id_bits(i) once the copy landed.
  __device__ __forceinline__ void copy_id(uint32_t dst, int64_t i) const;
  // read-only path (cached)
  __device__ __forceinline__ int64_t ldg(int64_t i) const {
    return i32 ? (int64_t)__ldg(static_cast<const int32_t*>(p) + i) : __ldg(static_cast<const int64_t*>(p) + i);
  }
};

__device__ __forceinline__ float ld_stream_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// x += a, y += b as one packed fp32x2 add (two IEEE round-to-nearest adds,
// bit-identical to two __fadd_rn, half the instructions).
__device__ __forceinline__ void add2(float& x, float& y, float a, float b) {
  asm("{\n\t.reg .b64 p, q;\n\t"
      "mov.b64 p, {%0, %1};\n\t"
      "mov.b64 q, {%2, %3};\n\t"
      "add.rn.f32x2 p, p, q;\n\t"
      "mov.b64 {%0, %1}, p;\n\t}"
      : "+f"(x), "+f"(y)
      : "f"(a), "f"(b));
}

// (a, b) * w as one packed fp32x2 multiply (each product rounded once).
__device__ __forceinline__ void mul2(float& a, float& b, float w) {
  asm("{\n\t.reg .b64 p, q;\n\t"
      "mov.b64 p, {%0, %1};\n\t"
      "mov.b64 q, {%2, %2};\n\t"
      "mul.rn.f32x2 p, p, q;\n\t"
      "mov.b64 {%0, %1}, p;\n\t}"
      : "+f"(a), "+f"(b)
      : "f"(w));
}

// Elements of a 16-byte chunk as floats.
template <int DT>
struct Chunk;

template <>
struct Chunk<TBE_F32> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void to_float(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

template <>
struct Chunk<TBE_F16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void to_float(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
      float2 p = __half22float2(h);
      f[2 * k] = p.x;
      f[2 * k + 1] = p.y;
    }
  }
};

template <>
struct Chunk<TBE_BF16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void to_float(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bf16 -> fp32 is exact: the bits move up 16 places
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
};

// Store n (4 or 8) floats rounded to the output type; `vec` selects vector
// stores (16 bytes, or 8 for four halves) when the destination is aligned.
template <typename OutT>
__device__ __forceinline__ void store_out(OutT* dst, const float* f, int n, bool vec);

template <>
__device__ __forceinline__ void store_out<float>(float* dst, const float* f, int n, bool vec) {
  if (vec) {
    for (int k = 0; k < n; k += 4)
      *reinterpret_cast<float4*>(dst + k) = make_float4(f[k], f[k + 1], f[k + 2], f[k + 3]);
  } else {
    for (int k = 0; k < n; ++k) dst[k] = f[k];
  }
}

template <>
__device__ __forceinline__ void store_out<__half>(__half* dst, const float* f, int n, bool vec) {
  if (vec && n == 8) {
    uint4 v;
    __half2 h0 = __floats2half2_rn(f[0], f[1]), h1 = __floats2half2_rn(f[2], f[3]);
    __half2 h2 = __floats2half2_rn(f[4], f[5]), h3 = __floats2half2_rn(f[6], f[7]);
    v.x = *reinterpret_cast<uint32_t*>(&h0);
    v.y = *reinterpret_cast<uint32_t*>(&h1);
    v.z = *reinterpret_cast<uint32_t*>(&h2);
    v.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(dst) = v;
  } else if (vec && n == 4) {
    __half2 h0 = __floats2half2_rn(f[0], f[1]), h1 = __floats2half2_rn(f[2], f[3]);
    *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
  } else {
    for (int k = 0; k < n; ++k) dst[k] = __float2half_rn(f[k]);
  }
}

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* dst, const float* f, int n,
                                                         bool vec) {
  if (vec && n == 8) {
    uint4 v;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(f[0], f[1]), h1 = __floats2bfloat162_rn(f[2], f[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(f[4], f[5]), h3 = __floats2bfloat162_rn(f[6], f[7]);
    v.x = *reinterpret_cast<uint32_t*>(&h0);
    v.y = *reinterpret_cast<uint32_t*>(&h1);
    v.z = *reinterpret_cast<uint32_t*>(&h2);
    v.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(dst) = v;
  } else if (vec && n == 4) {
    __nv_bfloat162 h0 = __floats2bfloat162_rn(f[0], f[1]), h1 = __floats2bfloat162_rn(f[2], f[3]);
    *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
  } else {
    for (int k = 0; k < n; ++k) dst[k] = __float2bfloat16_rn(f[k]);
  }
}


// ---------------------------------------------------------------------------
// asynchronous copies into shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the N most recent groups of this thread have landed
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void IdxPtr::copy_id(uint32_t dst, int64_t i) const {
  if (i32) {
    asm volatile("st.shared.u32 [%0+4], %1;" ::"r"(dst), "r"(0u) : "memory");
    cp_async4(dst, static_cast<const int32_t*>(p) + i);
  } else {
    cp_async8(dst, static_cast<const int64_t*>(p) + i);
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}


// ---------------------------------------------------------------------------
// bounded waits (every wait in the library gives up after a number of polls
// and lets the caller report TBE_DEV_TIMEOUT; no kernel waits forever)
// ---------------------------------------------------------------------------

// Polls *p (relaxed, GPU scope) until (*p & mask) != 0; returns the word, or
// 0 after `limit` polls.
__device__ inline uint32_t poll_word(const uint32_t* p, uint32_t mask, int limit) {
  for (int it = 0; it < limit; ++it) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v & mask) return v;
    if (it > 64) __nanosleep(100);
  }
  return 0;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Waits for phase `parity` of the shared-memory barrier; false after `limit`
// polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int limit) {
  const uint32_t a = smem_u32(bar);
  for (int it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}


// ---------------------------------------------------------------------------
// exact optimizer arithmetic (shared by the update kernel and the backward's
// fused update, so the two give bit-identical weights and momenta)
// ---------------------------------------------------------------------------

// Four consecutive elements of a table row of dtype dt, as floats and back
// (stores round to nearest-even); p is 16-byte aligned for fp32, 8 for halves.
__device__ __forceinline__ float4 load_quad(int dt, const uint8_t* p) {
  if (dt == TBE_F32) return *reinterpret_cast<const float4*>(p);
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  if (dt == TBE_F16) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),  // bf16: exact
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ void store_quad(int dt, uint8_t* p, float4 v) {
  if (dt == TBE_F32) {
    *reinterpret_cast<float4*>(p) = v;
    return;
  }
  uint2 u;
  if (dt == TBE_F16) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
  }
  *reinterpret_cast<uint2*>(p) = u;
}

// w - step * g, element by element, each one fused multiply-add.
__device__ __forceinline__ float4 fma_quad(float step, float4 g, float4 w) {
  w.x = fmaf(-step, g.x, w.x);
  w.y = fmaf(-step, g.y, w.y);
  w.z = fmaf(-step, g.z, w.z);
  w.w = fmaf(-step, g.w, w.w);
  return w;
}

// acc + the squares of the quad's elements (fused multiply-adds in order).
__device__ __forceinline__ float sum_sq(float4 v, float acc) {
  acc = fmaf(v.x, v.x, acc);
  acc = fmaf(v.y, v.y, acc);
  acc = fmaf(v.z, v.z, acc);
  return fmaf(v.w, v.w, acc);
}

// Sum over the warp by an xor butterfly (offsets 16, 8, 4, 2, 1).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Row-wise Adagrad: new momentum m + ss / D and the step lr / (sqrt(m') + eps),
// each operation rounded once (fp32).
__device__ __forceinline__ float adagrad_step(float lr, float eps, float m_old, float ss, int D, float* m_new) {
  *m_new = __fadd_rn(m_old, __fdiv_rn(ss, (float)D));
  return __fdiv_rn(lr, __fadd_rn(__fsqrt_rn(*m_new), eps));
}

// ---------------------------------------------------------------------------
// launchers (host)
// ---------------------------------------------------------------------------

struct FwdArgs {
  const uint8_t* weights;
  const TableMeta* meta;
  IdxPtr indices;
  IdxPtr offsets;
  const float* psw;
  void* out;
  int32_t* status;
  int32_t T;
  int32_t B;
  int64_t N;
  int32_t sumD;
  int32_t out_vec_ok;
  int32_t lpr_max;  // lanes per row cap of the gather (a power of two <= 32)
  int32_t balance;  // tables differ in shape: size each table's tasks by its own mean bag length
  int32_t mean;     // mean pooling: each bag's sum divided by its number of lookups
  int32_t split;    // stream kernel: 1 when the layout allows split tasks (set where the kernel is
                    // chosen); the launch replaces it by the bags per block (0: tasks per warp)
};

// Mean pooling: the bag's fp32 sum divided by its number of lookups, one IEEE
// division per element (the count is exact in fp32); an empty bag stays 0.
__device__ __forceinline__ void mean_scale(float* v, int n, int64_t len) {
  if (len > 0) {
    const float d = (float)len;
#pragma unroll
    for (int e = 0; e < n; ++e) v[e] = __fdiv_rn(v[e], d);
  }
}

int launch_forward_gather(const Plan& p, const FwdArgs& a, cudaStream_t s);
int launch_forward_histogram(const Plan& p, const FwdArgs& a, int32_t* counts_out, cudaStream_t s);

struct BwdArgs {
  const float* grad_out;
  const TableMeta* meta;
  IdxPtr indices;
  IdxPtr offsets;
  const float* psw;
  int64_t* unique_rows;
  int32_t* run_starts;
  int32_t* sorted_positions;
  float* row_grads;
  int64_t row_grads_capacity;
  int64_t* unique_count;
  void* workspace;
  size_t workspace_bytes;
  int32_t* status;
  int32_t T;
  int32_t B;
  int64_t N;
  int32_t sumD;
  // fused exact optimizer: opt_kind TBE_OPT_* or -1 (row gradients are stored)
  int32_t opt_kind;
  float lr, eps;
  uint8_t* weights;
  float* momentum;
};

size_t backward_workspace_bytes(const Plan& p, int32_t B, int64_t N);
constexpr int kBwdIndex = 1;   // backward stages that read only ids, offsets and weights
constexpr int kBwdReduce = 2;  // the reduction (reads grad_out)
int launch_backward(const Plan& p, const BwdArgs& a, cudaStream_t s, int stages = kBwdIndex | kBwdReduce);

struct UpdArgs {
  uint8_t* weights;
  const TableMeta* meta;
  float* momentum;
  const int64_t* unique_rows;
  const float* row_grads;
  const int64_t* unique_count;
  int64_t max_unique;
  int64_t row_grads_capacity;
  int32_t* status;
  int32_t T;
  int32_t kind;
  float lr;
  float eps;
};

int launch_exact_update(const Plan& p, const UpdArgs& a, cudaStream_t s);

}  // namespace tbe
