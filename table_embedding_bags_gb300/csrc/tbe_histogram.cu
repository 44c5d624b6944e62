// tbe_histogram.cu -- small-table forward: per-bag id histograms times the table
// on the 5th-generation tensor cores (tcgen05, accumulator in TMEM).
//
// [FBT] = the page "FBTriton table-batched embeddings: the backward win is a
// threshold moved from 32 to 256", section "The forward: a general gather and
// one clever special case": a pooled sum is a count-weighted sum of table
// rows, so for a table small enough to sit in one tile the pooled outputs of
// a group of bags are the matrix product counts[bags, rows] x table[rows, D].
// The page's kernel takes one unweighted fp16 table; this one takes every
// table of a plan whose tables are all small (at most 64 rows, D a multiple
// of 16 up to 256, fp16 or bf16), weighted or not, in one launch.
//
// Design (sm_103a), one CTA of 256 threads per tile of 128 bags of one table;
// the tiles are ordered table-major and each persistent CTA takes one
// contiguous range of them, so it loads a table into shared memory (the B
// operand, K-major) only when its range crosses into the next table.
//   1. Histogram.  Unweighted: all threads stream the tile's ids (one
//      contiguous range of `indices`) with coalesced loads and add 1 to the
//      bag's row in a shared-memory int32 histogram.  Weighted: the "count" of
//      (bag, row) is the sum of the per-sample weights of the bag's lookups of
//      that row, in fp32; a warp owns a bag and reads it 32 lookups at a time,
//      lanes holding the same row are summed in lane (= position) order by
//      the lowest of them, which then adds the sum to the cell: the
//      accumulation order is fixed, so the result does not depend on timing.
//   2. The A operand, per mode (A and B of one MMA always share a type):
//      * fp16 table:  counts as fp16, exact up to 2048;
//      * bf16 table:  counts are exact in bf16 only up to 256, so each count c
//        is split as lo = c mod 256 and hi = c - lo (a multiple of 256 up to
//        2048, exact too) and A = [lo | hi] runs two passes over K against
//        the same B tile;
//      * weighted:    the fp32 sum s is split into two tf32 terms
//        s1 = tf32(s), s2 = tf32(s - s1) (|s - s1 - s2| <= 2^-22 |s|),
//        A = [s1 | s2] and the table is widened to fp32 (exact for fp16 and
//        bf16 values), multiplied with kind::tf32.
//      Every product of a count term and a table value is exact in fp32; the
//      tensor core accumulates them in fp32.
//   3. One thread issues the MMAs (M = 128, N = D, fp32 accumulate in TMEM)
//      and commits them to an mbarrier; every wait on it is bounded.
//   4. Four warp pairs read the accumulator back with tcgen05.ld (each warp
//      reads its 32-lane TMEM quarter, the pair splits the columns), round
//      once to the output type and store.  An unweighted bag longer than 2048
//      ids (where a count may not fit its 16-bit form) is recomputed from the
//      int32 counts.
#include <algorithm>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kM = 128;                // bags per tile (MMA M)
constexpr int kMaxK = 64;              // table rows, padded to a multiple of 16
constexpr uint32_t kExactCount = 2048; // largest count both 16-bit count forms hold exactly
constexpr int kWaitLimit = 1 << 24;    // mbarrier polls before giving up (TBE_DEV_TIMEOUT)

// What a tile multiplies: the MMA kind and the form of its counts.
enum HistMode : int { kModeF16 = 0, kModeBF16 = 1, kModeTF32 = 2 };

// Dynamic shared memory of one CTA (offsets from a 1024-byte aligned base).
//   [0, 64 KB)   unweighted: int32 counts [kM][kMaxK] then the 16-bit A tile
//                [kM x 2K]; weighted: the tf32 A tile [kM x 2K], whose first K
//                columns accumulate the fp32 sums before they are split
//   b_tile       the table, [D x K] 16-bit or fp32, sized for the widest table
struct HistLayout {
  uint32_t counts, a16, b_tile, off, over, stage, mbar, tmem, total;
  __host__ __device__ HistLayout(int maxD, int b_esz) {
    counts = 0;
    a16 = kM * kMaxK * 4;
    b_tile = 2 * kM * kMaxK * 4;
    off = b_tile + ((maxD * kMaxK * b_esz + 1023) & ~1023);  // int64 [kM + 1]
    over = off + (kM + 1) * 8;                                // uint32 [kM / 32]
    stage = over + (kM / 32) * 4;                             // float [kWarps][32]
    mbar = (stage + kWarps * 32 * 4 + 7) & ~7u;               // uint64
    tmem = mbar + 8;                                          // uint32
    total = tmem + 8;
  }
};

// Canonical K-major layout without swizzle, in bytes: element (row, k) of an
// operand with `rows` rows and `esz`-byte elements sits in the 8-row x 16-byte
// core matrix (row / 8, k * esz / 16); core matrices are stored 8-row group
// first, so SBO = 128 bytes and LBO = (rows / 8) * 128 bytes.
__device__ __forceinline__ int kmajor_byte(int row, int k, int rows, int esz) {
  const int kb = k * esz;
  return (((kb >> 4) * (rows >> 3) + (row >> 3)) << 7) + ((row & 7) << 4) + (kb & 15);
}

// tcgen05 shared-memory matrix descriptor (no swizzle, version 1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3fff) | ((uint64_t)((lbo >> 4) & 0x3fff) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fff) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16 / kind::tf32: A and B K-major of
// format fmt (0 = fp16, 1 = bf16, 2 = tf32), fp32 D, M = 128, N = n.
__device__ __forceinline__ uint32_t instr_desc(int fmt, int n) {
  return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kM >> 4) << 24);
}

// Round to the nearest tf32 value (10 fraction bits, ties to even), as fp32
// bits with the 13 low fraction bits zero.  Finite inputs only.
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0xfffu + ((u >> 13) & 1u);
  return __uint_as_float(u & 0xffffe000u);
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

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
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

// Launch-wide shape of the histogram path.
struct HistShape {
  int32_t maxD;   // widest table (sizes the B tile and the TMEM accumulator)
  int32_t b_esz;  // 4 when some tile may take the weighted (tf32) form, else 2
  int32_t tpt;    // tiles per table, ceil(B / kM)
};

// A table element as fp32 (fp16 or bf16 storage).
__device__ __forceinline__ float table_value(uint16_t bits, int dtype) {
  return dtype == TBE_F16 ? __half2float(__ushort_as_half(bits)) : __bfloat162float(__ushort_as_bfloat16(bits));
}

// The tile's table into the B tile: element (n = column d, k = row r) = W[r][d];
// rows r >= rows (the K padding) are zero.
__device__ void load_table(unsigned char* b_tile, const uint16_t* table, int rows, int K, int D, int dtype,
                           int mode, int tid) {
  for (int e = tid; e < D * K; e += kThreads) {
    const int r = e / D, d = e - r * D;
    const uint16_t bits = r < rows ? table[(int64_t)r * D + d] : (uint16_t)0;
    if (mode == kModeTF32)
      *reinterpret_cast<float*>(b_tile + kmajor_byte(d, r, D, 4)) = r < rows ? table_value(bits, dtype) : 0.f;
    else
      *reinterpret_cast<uint16_t*>(b_tile + kmajor_byte(d, r, D, 2)) = bits;
  }
}

template <typename OutT, bool COUNTS_ONLY>
__global__ void __launch_bounds__(kThreads, 2) hist_kernel(const FwdArgs a, const HistShape h, int32_t* counts_out) {
  extern __shared__ unsigned char smem_raw[];
  const HistLayout L(h.maxD, h.b_esz);
  unsigned char* base = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  int32_t* counts = reinterpret_cast<int32_t*>(base + L.counts);
  unsigned char* a32 = base + L.counts;  // the tf32 A tile shares the counts region
  unsigned char* a16 = base + L.a16;
  unsigned char* b_tile = base + L.b_tile;
  int64_t* off = reinterpret_cast<int64_t*>(base + L.off);
  uint32_t* over = reinterpret_cast<uint32_t*>(base + L.over);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(base + L.mbar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* stage = reinterpret_cast<float*>(base + L.stage) + warp * 32;
  const uint32_t ncols = h.maxD <= 32 ? 32 : (h.maxD <= 64 ? 64 : (h.maxD <= 128 ? 128 : 256));  // TMEM columns
  const int64_t ntiles = (int64_t)a.T * h.tpt;
  const int64_t TB = (int64_t)a.T * a.B;
  const int64_t tile_begin = ntiles * blockIdx.x / gridDim.x;
  const int64_t tile_end = ntiles * (blockIdx.x + 1) / gridDim.x;

  if (!COUNTS_ONLY) {
    if (warp == 0) tmem_alloc(tmem_slot, ncols);
    if (tid == 0) mbar_init(mbar);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  }
  __syncthreads();
  const uint32_t tmem = COUNTS_ONLY ? 0u : *tmem_slot;
  uint32_t phase = 0;
  int cur_t = -1, cur_mode = -1;

  for (int64_t tile = tile_begin; tile < tile_end; ++tile) {
    const int t = (int)(tile / h.tpt);
    const int b0 = (int)(tile - (int64_t)t * h.tpt) * kM;
    const int nbag = min(kM, a.B - b0);
    const TableMeta m = a.meta[t];
    const int rows = m.rows, D = m.D;
    const int K = (rows + 15) & ~15;  // MMA K, padded to 16
    const bool weighted = !COUNTS_ONLY && a.psw != nullptr && m.weighted;
    const int mode = weighted ? kModeTF32 : (m.dtype == TBE_F16 ? kModeF16 : kModeBF16);
    const int64_t g0 = (int64_t)t * a.B + b0;

    if (weighted) {
      for (int e = tid; e < K * (kM * 4 / 16); e += kThreads) reinterpret_cast<int4*>(a32)[e] = make_int4(0, 0, 0, 0);
    } else {
      for (int e = tid; e < kM * kMaxK / 4; e += kThreads) reinterpret_cast<int4*>(counts)[e] = make_int4(0, 0, 0, 0);
    }
    if (tid < kM / 32) over[tid] = 0;
    for (int q = tid; q <= nbag; q += kThreads) off[q] = a.offsets.stream(g0 + q);
    if (!COUNTS_ONLY && (t != cur_t || mode != cur_mode)) {
      load_table(b_tile, reinterpret_cast<const uint16_t*>(a.weights + m.w_off), rows, K, D, m.dtype, mode, tid);
      cur_t = t;
      cur_mode = mode;
    }
    __syncthreads();
    {
      // bag bounds: must start at 0, never decrease and end at N; a broken
      // tile is reported and pooled as empty
      int bad = off[0] < 0 || off[nbag] > a.N || (g0 == 0 && off[0] != 0) || (g0 + nbag == TB && off[nbag] != a.N);
      for (int q = tid; q < nbag; q += kThreads) bad |= off[q + 1] < off[q];
      bad = __syncthreads_or(bad);
      if (bad) {
        if (tid == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
        for (int q = tid; q <= nbag; q += kThreads) off[q] = 0;
      }
      __syncthreads();
    }

    bool bad_id = false;
    const int64_t p0 = off[0], p1 = off[nbag];
    if (!weighted) {
      // counts of every bag of the tile; a thread's positions only grow, so
      // its bag index only moves forward
      int q = 0;
      {
        const int64_t p = p0 + tid;
        int lo = 0, hi = nbag - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (off[mid] <= p) lo = mid; else hi = mid - 1;
        }
        q = lo;
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
          while (q < nbag - 1 && off[q + 1] <= p) ++q;
          if ((uint64_t)id[u] < (uint64_t)rows) atomicAdd(&counts[q * kMaxK + (int)id[u]], 1);
          else bad_id = true;
        }
      }
      for (int b = tid; b < nbag; b += kThreads)
        if (off[b + 1] - off[b] > (int64_t)kExactCount) atomicOr(&over[b >> 5], 1u << (b & 31));
    } else {
      // sums of per-sample weights: warp per bag, 32 lookups per step in
      // position order; lanes holding the same row are summed in lane order
      // by the lowest of them, which alone adds to the cell
      constexpr int kWU = 4;
      for (int q = warp; q < nbag; q += kWarps) {
        const int64_t s = off[q], e = off[q + 1];
        for (int64_t pb = s; pb < e; pb += 32 * kWU) {
          int64_t id[kWU];
          float w[kWU];
#pragma unroll
          for (int u = 0; u < kWU; ++u) {
            const int64_t p = pb + u * 32 + lane;
            id[u] = p < e ? a.indices.stream(p) : -1;
            w[u] = p < e ? __ldg(a.psw + p) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < kWU; ++u) {
            if (pb + u * 32 >= e) break;  // warp-uniform
            const bool in = pb + u * 32 + lane < e;
            const bool ok = in && (uint64_t)id[u] < (uint64_t)rows;
            bad_id |= in && !ok;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? (unsigned long long)id[u] : ~0ull);
            stage[lane] = w[u];
            __syncwarp();
            if (ok && __ffs(peers) - 1 == lane) {
              float sum = 0.f;
              for (unsigned mm = peers; mm; mm &= mm - 1) sum += stage[__ffs(mm) - 1];
              *reinterpret_cast<float*>(a32 + kmajor_byte(q, (int)id[u], kM, 4)) += sum;
            }
            __syncwarp();
          }
        }
      }
    }
    if (bad_id) report(a.status, TBE_DEV_BAD_INDEX);
    __syncthreads();

    if (COUNTS_ONLY) {
      int32_t* dst = counts_out + m.row_base * (int64_t)a.B + (int64_t)b0 * rows;
      for (int e = tid; e < nbag * rows; e += kThreads) {
        const int q = e / rows, r = e - q * rows;
        dst[e] = counts[q * kMaxK + r];
      }
      __syncthreads();
      continue;
    }

    // the A operand (see the header: one or two K passes per mode)
    if (mode == kModeTF32) {
      for (int e = tid; e < kM * K; e += kThreads) {
        const int q = e / K, r = e - q * K;
        float* cell = reinterpret_cast<float*>(a32 + kmajor_byte(q, r, kM, 4));
        const float s = *cell, s1 = round_tf32(s);
        *cell = s1;
        *reinterpret_cast<float*>(a32 + kmajor_byte(q, K + r, kM, 4)) = round_tf32(s - s1);
      }
    } else if (mode == kModeF16) {
      for (int e = tid; e < kM * K; e += kThreads) {
        const int q = e / K, r = e - q * K;
        const int32_t c = min(counts[q * kMaxK + r], (int32_t)kExactCount);
        *reinterpret_cast<__half*>(a16 + kmajor_byte(q, r, kM, 2)) = __int2half_rn(c);
      }
    } else {
      for (int e = tid; e < kM * K; e += kThreads) {
        const int q = e / K, r = e - q * K;
        const int32_t c = min(counts[q * kMaxK + r], (int32_t)kExactCount), lo = c & 255;
        *reinterpret_cast<__nv_bfloat16*>(a16 + kmajor_byte(q, r, kM, 2)) = __float2bfloat16_rn((float)lo);
        *reinterpret_cast<__nv_bfloat16*>(a16 + kmajor_byte(q, K + r, kM, 2)) = __float2bfloat16_rn((float)(c - lo));
      }
    }
    // make the generic-proxy shared-memory writes visible to the tensor core
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int esz = mode == kModeTF32 ? 4 : 2;
      const uint32_t idesc = instr_desc(mode, D);  // the mode values are the descriptor's formats
      const int a_steps = (mode == kModeF16 ? K : 2 * K) * esz / 32;  // 32 bytes of K per MMA
      const int b_steps = K * esz / 32;
      const uint32_t a_addr = smem_u32(mode == kModeTF32 ? a32 : a16), b_addr = smem_u32(b_tile);
      for (int st = 0; st < a_steps; ++st) {
        // step st covers core-matrix columns 2st and 2st+1 (LBO apart); the
        // second pass over K reuses the B steps
        const int sb = st % b_steps;
        const uint64_t ad = smem_desc(a_addr + st * 2 * (kM / 8) * 128, (kM / 8) * 128, 128);
        const uint64_t bd = smem_desc(b_addr + sb * 2 * (D / 8) * 128, (D / 8) * 128, 128);
        if (mode == kModeTF32) mma_tf32(tmem, ad, bd, idesc, st > 0 ? 1u : 0u);
        else mma_f16(tmem, ad, bd, idesc, st > 0 ? 1u : 0u);
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
      OutT* orow = reinterpret_cast<OutT*>(a.out) + (int64_t)(b0 + q) * a.sumD + m.col_off;
      const int ngroups = (D + 31) / 32;
      const int per_warp = (ngroups + 1) / 2;
      const bool vec = a.out_vec_ok;
      for (int gq = 0; gq < per_warp; ++gq) {
        const int cg = (warp >> 2) * per_warp + gq;
        if (cg >= ngroups) break;
        float v[32];
        tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(cg * 32), v);
        if (is_over) {  // exact recount of an unweighted bag too long for 16-bit counts
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (cg * 32 + c < D) {
              float acc = 0.f;
              for (int r = 0; r < rows; ++r) {
                const uint16_t bits = *reinterpret_cast<const uint16_t*>(b_tile + kmajor_byte(cg * 32 + c, r, D, 2));
                acc = __fadd_rn(acc, __fmul_rn((float)counts[q * kMaxK + r], table_value(bits, m.dtype)));
              }
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
int launch_hist(const FwdArgs& a, const HistShape& h, int32_t* counts, cudaStream_t s) {
  const size_t smem = HistLayout(h.maxD, h.b_esz).total + 1024;  // + alignment slack
  if (cudaFuncSetAttribute(hist_kernel<OutT, COUNTS_ONLY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(hist_kernel<OutT, COUNTS_ONLY>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return TBE_ERR_CUDA;
  const int64_t ntiles = (int64_t)a.T * h.tpt;
  // CTAs per SM from the kernel's registers and shared memory (the launch
  // bounds keep it at <= 128 registers, so two fit the register file),
  // capped so that their TMEM accumulators fit the 512 columns of an SM
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
  const int ncols = h.maxD <= 32 ? 32 : (h.maxD <= 64 ? 64 : (h.maxD <= 128 ? 128 : 256));
  if (!COUNTS_ONLY) per_sm = std::min(per_sm, 512 / ncols);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ntiles, (int64_t)sm_count() * per_sm));
  hist_kernel<OutT, COUNTS_ONLY><<<grid, kThreads, smem, s>>>(a, h, counts);
  return check_launch();
}

}  // namespace

int launch_forward_histogram(const Plan& p, const FwdArgs& a, int32_t* counts_out, cudaStream_t s) {
  HistShape h;
  h.maxD = p.maxD;
  h.b_esz = (!counts_out && a.psw != nullptr && p.any_weighted) ? 4 : 2;
  h.tpt = (a.B + kM - 1) / kM;
  if (counts_out) return launch_hist<float, true>(a, h, counts_out, s);
  switch (p.out_dtype) {
    case TBE_F32: return launch_hist<float, false>(a, h, nullptr, s);
    case TBE_F16: return launch_hist<__half, false>(a, h, nullptr, s);
    default: return launch_hist<__nv_bfloat16, false>(a, h, nullptr, s);
  }
}

}  // namespace tbe
