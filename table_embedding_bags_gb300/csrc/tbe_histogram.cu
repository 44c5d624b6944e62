// tbe_histogram.cu -- small-table forward: per-bag id histograms times the table
// on the 5th-generation tensor cores (tcgen05, accumulator in TMEM).
//
// [FBT] = the page "FBTriton table-batched embeddings: the backward win is a
// threshold moved from 32 to 256", section "The forward: a general gather and
// one clever special case": a pooled sum is a count-weighted sum of table
// rows, so for a table small enough to sit in one tile the pooled outputs of
// a group of bags are the matrix product counts[bags, rows] x table[rows, D];
// counts are exact in fp16 (every integer up to 2048 is an fp16 value).
//
// Design (sm_103a), one CTA of 256 threads per tile of 128 bags (persistent):
//   1. H2: the tile's ids are one contiguous range of `indices`; all threads
//      stream it with coalesced loads and add each id to its bag's row in a
//      shared-memory int32 histogram (the bag of a position is found in the
//      tile's 129 offsets staged in shared memory).
//   2. The counts are written as an fp16 A tile [128 x K] and the table (once
//      per CTA) as an fp16 B tile [K x D] in the canonical K-major layout
//      without swizzle (8 x 16-byte core matrices; SBO = distance between
//      8-row groups, LBO = distance between core matrices along K).
//   3. H3: one thread issues K/16 tcgen05.mma.cta_group::1.kind::f16
//      (M = 128, N = D, fp32 accumulate in TMEM) and commits them to an
//      mbarrier; every wait on it is bounded.
//   4. Four warp pairs read the accumulator back with tcgen05.ld (each warp
//      reads its 32-lane TMEM quarter, the pair splits the columns), round
//      once to the output type and store.  A bag longer than 2048 ids (where
//      fp16 counts may stop being exact) is recomputed from the int32 counts.
#include <algorithm>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kThreads = 256;
constexpr int kM = 128;                // bags per tile (MMA M)
constexpr int kMaxK = 64;              // table rows, padded to a multiple of 16
constexpr uint32_t kExactCount = 2048; // largest count every fp16 value can hold exactly
constexpr int kWaitLimit = 1 << 24;    // mbarrier polls before giving up (TBE_DEV_TIMEOUT)

// Dynamic shared memory of one CTA (offsets from a 1024-byte aligned base).
struct HistLayout {
  uint32_t counts, a_tile, b_tile, off, over, mbar, tmem, total;
  __host__ __device__ HistLayout(int D) {
    const int K = kMaxK;
    counts = 0;                                       // int32 [kM][kMaxK]
    a_tile = counts + kM * kMaxK * 4;                 // fp16 [kM][K] canonical K-major
    b_tile = a_tile + kM * K * 2;                     // fp16 [D][K] canonical K-major
    off = b_tile + ((D * K * 2 + 1023) & ~1023);      // int64 [kM + 1]
    over = off + (kM + 1) * 8;                        // uint32 [kM / 32]
    mbar = (over + (kM / 32) * 4 + 7) & ~7u;          // uint64
    tmem = mbar + 8;                                  // uint32
    total = tmem + 8;
  }
};


// Canonical K-major layout without swizzle: element (row, k) of an operand
// with `rows` rows sits in core matrix (row / 8, k / 8); core matrices are
// stored 8-row group first, so SBO = 128 bytes and LBO = (rows / 8) * 128.
__device__ __forceinline__ int kmajor_index(int row, int k, int rows) {
  return (((k >> 3) * (rows >> 3) + (row >> 3)) << 6) + ((row & 7) << 3) + (k & 7);
}

// tcgen05 shared-memory matrix descriptor (no swizzle, version 1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3fff) | ((uint64_t)((lbo >> 4) & 0x3fff) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fff) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp16 A and B (both K-major), fp32 D,
// M = 128, N = n.
__device__ __forceinline__ uint32_t instr_desc_f16(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
}


__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]);
}

template <typename OutT, bool COUNTS_ONLY>
__global__ void __launch_bounds__(kThreads, 2) hist_kernel(const FwdArgs a, int32_t* counts_out) {
  extern __shared__ unsigned char smem_raw[];
  const int D = __ldg(&a.meta[0].D);
  const HistLayout L(D);
  unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  int32_t* counts = reinterpret_cast<int32_t*>(base + L.counts);
  __half* a_tile = reinterpret_cast<__half*>(base + L.a_tile);
  __half* b_tile = reinterpret_cast<__half*>(base + L.b_tile);
  int64_t* off = reinterpret_cast<int64_t*>(base + L.off);
  uint32_t* over = reinterpret_cast<uint32_t*>(base + L.over);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(base + L.mbar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = (int)__ldg(&a.meta[0].rows);
  const int K = (rows + 15) & ~15;                      // MMA K, padded to 16
  const uint32_t ncols = D <= 32 ? 32 : (D <= 64 ? 64 : (D <= 128 ? 128 : 256));  // TMEM columns
  const int ntiles = (a.B + kM - 1) / kM;

  if (!COUNTS_ONLY) {
    if (warp == 0) tmem_alloc(tmem_slot, ncols);
    if (tid == 0) mbar_init(mbar);
    // the table as the B operand: element (n = column d, k = row r) = W[r][d]
    const __half* table = reinterpret_cast<const __half*>(a.weights + __ldg(&a.meta[0].w_off));
    for (int e = tid; e < D * K; e += kThreads) {
      const int r = e / D, d = e - r * D;
      b_tile[kmajor_index(d, r, D)] = r < rows ? table[(int64_t)r * D + d] : __float2half_rn(0.f);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  }
  __syncthreads();
  const uint32_t tmem = COUNTS_ONLY ? 0u : *tmem_slot;
  uint32_t phase = 0;

  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int b0 = tile * kM;
    const int nbag = min(kM, a.B - b0);
    for (int e = tid; e < kM * kMaxK / 4; e += kThreads) reinterpret_cast<int4*>(counts)[e] = make_int4(0, 0, 0, 0);
    if (tid < kM / 32) over[tid] = 0;
    // bag bounds (feature-major offsets of table 0): must start at 0, never
    // decrease and end at N; a broken tile is reported and pooled as empty
    for (int m = tid; m <= nbag; m += kThreads) off[m] = a.offsets.stream(b0 + m);
    __syncthreads();
    {
      int bad = off[0] < 0 || off[nbag] > a.N || (b0 == 0 && off[0] != 0) || (b0 + nbag == a.B && off[nbag] != a.N);
      for (int m = tid; m < nbag; m += kThreads) bad |= off[m + 1] < off[m];
      bad = __syncthreads_or(bad);
      if (bad) {
        if (tid == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
        for (int m = tid; m <= nbag; m += kThreads) off[m] = 0;
      }
      __syncthreads();
    }
    // H2: histogram of every bag of the tile; a thread's positions only grow,
    // so its bag index only moves forward
    const int64_t p0 = off[0], p1 = off[nbag];
    bool bad_id = false;
    int m = 0;
    {
      const int64_t p = p0 + tid;
      int lo = 0, hi = nbag - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= p) lo = mid; else hi = mid - 1;
      }
      m = lo;
    }
    constexpr int kU = 16;
    for (int64_t pb = p0; pb < p1; pb += kThreads * kU) {
      int64_t id[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t p = pb + u * kThreads + tid;
        id[u] = p < p1 ? a.indices.stream(p) : -1;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t p = pb + u * kThreads + tid;
        if (p >= p1) break;
        while (m < nbag - 1 && off[m + 1] <= p) ++m;
        if ((uint64_t)id[u] < (uint64_t)rows) atomicAdd(&counts[m * kMaxK + (int)id[u]], 1);
        else bad_id = true;
      }
    }
    if (bad_id) report(a.status, TBE_DEV_BAD_INDEX);
    for (int q = tid; q < nbag; q += kThreads)
      if (off[q + 1] - off[q] > (int64_t)kExactCount) atomicOr(&over[q >> 5], 1u << (q & 31));
    __syncthreads();

    if (COUNTS_ONLY) {
      for (int e = tid; e < nbag * rows; e += kThreads) {
        const int q = e / rows, r = e - q * rows;
        counts_out[(int64_t)(b0 + q) * rows + r] = counts[q * kMaxK + r];
      }
      __syncthreads();
      continue;
    }
    // counts -> fp16 A operand [128 x K] (exact up to 2048; longer bags are redone below)
    for (int e = tid; e < kM * K; e += kThreads) {
      const int q = e / K, r = e - q * K;
      const int32_t c = q < nbag ? counts[q * kMaxK + r] : 0;
      a_tile[kmajor_index(q, r, kM)] = __int2half_rn(min(c, (int32_t)kExactCount));
    }
    // make the generic-proxy shared-memory writes visible to the tensor core
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t idesc = instr_desc_f16(D);
      const uint32_t a_addr = smem_u32(a_tile), b_addr = smem_u32(b_tile);
      for (int ks = 0; ks < K / 16; ++ks) {
        // K step ks covers core-matrix columns 2ks and 2ks+1 (LBO apart)
        const uint64_t ad = smem_desc(a_addr + ks * 2 * (kM / 8) * 128, (kM / 8) * 128, 128);
        const uint64_t bd = smem_desc(b_addr + ks * 2 * (D / 8) * 128, (D / 8) * 128, 128);
        mma_f16(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
      mma_commit(mbar);
    }
    const bool ok = mbar_wait(mbar, phase, kWaitLimit);
    phase ^= 1u;
    if (__syncthreads_or(!ok)) {  // the whole CTA stops together
      if (tid == 0) report(a.status, TBE_DEV_TIMEOUT);
      break;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    {
      // epilogue: warp w reads TMEM lanes 32*(w%4).. (bags); warps w and w+4
      // split the 32-column groups
      const int q = (warp & 3) * 32 + lane;
      const bool is_over = q < nbag && ((over[q >> 5] >> (q & 31)) & 1u);
      OutT* orow = reinterpret_cast<OutT*>(a.out) + (int64_t)(b0 + q) * a.sumD + __ldg(&a.meta[0].col_off);
      const int ngroups = (D + 31) / 32;
      const int per_warp = (ngroups + 1) / 2;
      const bool vec = a.out_vec_ok;
      for (int gq = 0; gq < per_warp; ++gq) {
        const int cg = (warp >> 2) * per_warp + gq;
        if (cg >= ngroups) break;
        float v[32];
        tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(cg * 32), v);
        if (is_over) {  // exact recount for bags too long for fp16 counts
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (cg * 32 + c < D) {
              float acc = 0.f;
              for (int r = 0; r < rows; ++r)
                acc = __fadd_rn(acc, __fmul_rn((float)counts[q * kMaxK + r],
                                               __half2float(b_tile[kmajor_index(cg * 32 + c, r, D)])));
              v[c] = acc;
            }
          }
        }
        if (q < nbag) {
#pragma unroll
          for (int c = 0; c < 32; c += 8)
            if (cg * 32 + c < D) store_out<OutT>(orow + cg * 32 + c, v + c, 8, vec);
        }
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
  }
  if (!COUNTS_ONLY) {
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, ncols);
  }
}

template <typename OutT, bool COUNTS_ONLY>
int launch_hist(const FwdArgs& a, int32_t* counts, int D, cudaStream_t s) {
  const size_t smem = HistLayout(D).total + 1024;  // + alignment slack
  if (cudaFuncSetAttribute(hist_kernel<OutT, COUNTS_ONLY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(hist_kernel<OutT, COUNTS_ONLY>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return TBE_ERR_CUDA;
  const int ntiles = (a.B + kM - 1) / kM;
  // CTAs per SM: what shared memory allows, capped so that their TMEM
  // accumulators (<= 256 columns each) fit the 512 columns of an SM
  // CTAs per SM from the kernel's registers and shared memory (the launch
  // bounds keep it at <= 128 registers, so two fit the register file)
  int per_sm = 2;
  {
    cudaFuncAttributes fa;
    int dev = 0, smem_sm = 0;
    cudaGetDevice(&dev);
    if (cudaFuncGetAttributes(&fa, hist_kernel<OutT, COUNTS_ONLY>) == cudaSuccess &&
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess) {
      const int by_regs = 65536 / std::max(1, fa.numRegs * kThreads);
      const int by_smem = smem_sm / (int)(smem + 1024);
      per_sm = std::max(1, std::min(by_regs, by_smem));
    }
  }
  const int ncols = D <= 32 ? 32 : (D <= 64 ? 64 : (D <= 128 ? 128 : 256));
  if (!COUNTS_ONLY) per_sm = std::min(per_sm, 512 / ncols);
  const int grid = std::max(1, std::min(ntiles, sm_count() * per_sm));
  hist_kernel<OutT, COUNTS_ONLY><<<grid, kThreads, smem, s>>>(a, counts);
  return check_launch();
}

}  // namespace

int launch_forward_histogram(const Plan& p, const FwdArgs& a, int32_t* counts_out, cudaStream_t s) {
  const int D = p.hmeta[0].D;
  if (counts_out) return launch_hist<float, true>(a, counts_out, D, s);
  switch (p.out_dtype) {
    case TBE_F32: return launch_hist<float, false>(a, nullptr, D, s);
    case TBE_F16: return launch_hist<__half, false>(a, nullptr, D, s);
    default: return launch_hist<__nv_bfloat16, false>(a, nullptr, D, s);
  }
}

}  // namespace tbe
