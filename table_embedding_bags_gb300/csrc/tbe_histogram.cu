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

constexpr int kConsumers = 512;                 // threads that count, multiply and store
constexpr int kWarps = kConsumers / 32;         // consumer warps
constexpr int kProducers = 128;                 // threads streaming the ids into the ring
constexpr int kThreads = kConsumers + kProducers;
constexpr int kM = 128;                // bags per tile (MMA M)
constexpr int kMaxK = 64;              // table rows, padded to a multiple of 16
constexpr uint32_t kExactCount = 2048; // largest count both 16-bit count forms hold exactly
constexpr int kWaitLimit = 1 << 24;    // mbarrier polls before giving up (TBE_DEV_TIMEOUT)
constexpr int kChunk = 16384;          // bytes per id chunk (32 bytes per consumer thread)
constexpr int kRingMin = 2;            // chunks in the id ring: as many as shared memory leaves room for
constexpr int kRingMax = 24;
constexpr int kLut = 4096;             // bag of every 32nd position of a tile (tiles of up to 128 Ki ids)

// What a tile multiplies: the MMA kind and the form of its counts.
enum HistMode : int { kModeF16 = 0, kModeBF16 = 1, kModeTF32 = 2 };

// Dynamic shared memory of one CTA (offsets from a 1024-byte aligned base).
//   [0, 32 KB)   unweighted: int32 counts [kM][kMaxK]
//   [32, 64 KB)  the 16-bit A tile [kM x 2K].  Weighted tiles use [0, 64 KB)
//                as the tf32 A tile [kM x 2K], whose first K columns
//                accumulate the fp32 sums before they are split.
//   b_tile       the table, [D x K] 16-bit or fp32, sized for the widest table
//   ring         `ring` chunks of kChunk bytes of ids
struct HistLayout {
  uint32_t counts, a16, b_tile, ring, off, over, stage, mbar, tmem, flags, total;
  __host__ __device__ HistLayout(int maxD, int b_esz, int nring) {
    counts = 0;
    a16 = kM * kMaxK * 4;
    b_tile = 2 * kM * kMaxK * 4;
    ring = b_tile + ((maxD * kMaxK * b_esz + 1023) & ~1023);
    off = ring + nring * kChunk;                              // int64 [kM + 1]
    over = off + (kM + 1) * 8;  // uint32 [kM / 32]; then int32 off32 [kM + 1], uint8 lut [kLut]
    stage = over + (kM / 32) * 4 + ((kM + 1) * 4 + 15) / 16 * 16 + kLut;  // float [kWarps][32]
    mbar = (stage + kWarps * 32 * 4 + 7) & ~7u;               // uint64: MMA, full[kRingMax], empty[kRingMax]
    tmem = mbar + 8 * (1 + 2 * kRingMax);                     // uint32
    flags = tmem + 4;                                         // int32 [4]: [0] stop
    total = flags + 16;
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

constexpr int kRun = kChunk / kConsumers;  // bytes of a chunk one consumer thread counts
static_assert(kRun == 32, "a chunk is one 32-byte run per consumer thread");

__device__ __forceinline__ void mbar_init_count(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier 1 over the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ int consumers_sync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred), "n"(kConsumers)
      : "memory");
  return r;
}

// The ids a tile streams through the ring: the 16-byte aligned middle of its
// range [p0, p1) (clamped to [0, N]), cut into chunks; the ragged ends (under
// 16 bytes each) are read directly.  Producer and consumers derive it from
// the same two offsets, so they agree on every chunk.
struct ChunkPlan {
  uintptr_t beg, end;  // aligned byte range
  int64_t p0, p1;      // the tile's positions
  int64_t pa, pe;      // first position of the aligned middle / of the ragged tail
  int nch;             // chunks
  __device__ ChunkPlan(const void* ids, int w, int64_t r0, int64_t r1, int64_t N) {
    p0 = min(max(r0, (int64_t)0), N);
    p1 = min(max(r1, p0), N);
    const uintptr_t src0 = (uintptr_t)ids + (uintptr_t)(p0 * w), src1 = (uintptr_t)ids + (uintptr_t)(p1 * w);
    beg = min((src0 + 15) & ~(uintptr_t)15, src1);
    end = max(src1 & ~(uintptr_t)15, beg);
    pa = p0 + (int64_t)((beg - src0) / w);
    pe = p0 + (int64_t)((end - src0) / w);
    nch = (int)((end - beg + kChunk - 1) / kChunk);
  }
  __device__ uint32_t bytes(int c) const { return (uint32_t)min((uintptr_t)kChunk, end - beg - (uintptr_t)c * kChunk); }
};

// Bag of position p within a tile: the last q < nbag with off[q] <= p.
__device__ __forceinline__ int tile_bag(const int64_t* off, int nbag, int64_t p) {
  int lo = 0, hi = nbag - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= p) lo = mid; else hi = mid - 1;
  }
  return lo;
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
  int32_t mb;     // bags per tile (<= kM; rows nbag..kM-1 of the MMA are zero)
  int32_t tpt;    // tiles per table, ceil(B / mb)
  int32_t ring;   // chunks in the id ring (kRingMin .. kRingMax)
};

// A table element as fp32 (fp16 or bf16 storage).
__device__ __forceinline__ float table_value(uint16_t bits, int dtype) {
  return dtype == TBE_F16 ? __half2float(__ushort_as_half(bits)) : __bfloat162float(__ushort_as_bfloat16(bits));
}

// The tile's table into the B tile: element (n = column d, k = row r) = W[r][d];
// rows r >= rows (the K padding) are zero.  The table is read as 16-byte
// chunks (8 elements of a row), all of a thread's chunks in flight at once.
__device__ void load_table(unsigned char* b_tile, const unsigned char* table, int rows, int K, int D, int dtype,
                           int mode, int tid) {
  constexpr int kPer = kMaxK * 256 / 8 / kConsumers;  // chunks per thread of the largest table
  const int cpr = D >> 3;                           // chunks per row
  const int n = rows * cpr;
  uint4 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * kConsumers;
    if (e < n) v[u] = __ldg(reinterpret_cast<const uint4*>(table) + e);
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * kConsumers;
    if (e >= n) break;
    const int r = e / cpr, d0 = (e - r * cpr) << 3;
    const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint16_t bits = (uint16_t)(w4[k >> 1] >> ((k & 1) * 16));
      if (mode == kModeTF32)
        *reinterpret_cast<float*>(b_tile + kmajor_byte(d0 + k, r, D, 4)) = table_value(bits, dtype);
      else
        *reinterpret_cast<uint16_t*>(b_tile + kmajor_byte(d0 + k, r, D, 2)) = bits;
    }
  }
  for (int e = tid; e < (K - rows) * D; e += kConsumers) {
    const int r = rows + e / D, d = e - (r - rows) * D;
    if (mode == kModeTF32) *reinterpret_cast<float*>(b_tile + kmajor_byte(d, r, D, 4)) = 0.f;
    else *reinterpret_cast<uint16_t*>(b_tile + kmajor_byte(d, r, D, 2)) = 0;
  }
}

// Two adjacent outputs rounded to the output type (one 8- or 4-byte store
// when the row segment is 16-byte aligned).
template <typename OutT>
__device__ __forceinline__ void store_pair(OutT* dst, float x, float y, bool vec);

template <>
__device__ __forceinline__ void store_pair<float>(float* dst, float x, float y, bool vec) {
  if (vec) *reinterpret_cast<float2*>(dst) = make_float2(x, y);
  else { dst[0] = x; dst[1] = y; }
}

template <>
__device__ __forceinline__ void store_pair<__half>(__half* dst, float x, float y, bool vec) {
  if (vec) *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(x, y);
  else { dst[0] = __float2half_rn(x); dst[1] = __float2half_rn(y); }
}

template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16* dst, float x, float y, bool vec) {
  if (vec) *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(x, y);
  else { dst[0] = __float2bfloat16_rn(x); dst[1] = __float2bfloat16_rn(y); }
}

// Counts this thread's runs of the tile's staged id chunks: of each chunk,
// the kRun bytes at tid * kRun (4 int64 or 8 int32 ids), and releases each
// chunk (per warp) when done.  Positions are relative to the tile's first
// id, in 32 bits.  The bag of a run's first position comes from the tile's
// lookup of every 32nd position (lut, when the tile has one) or from the
// previous run, and moves forward past the bag starts up to it.  Returns
// false when a chunk never arrived (decided per warp).
template <int W>
__device__ __forceinline__ bool consume_chunks(const unsigned char* ring, uint64_t* full, uint64_t* empty, int R,
                                               uint32_t& slot, uint32_t& par, int nch, uint32_t last_bytes,
                                               int32_t pa, bool count, const int32_t* off32, const uint8_t* lut,
                                               int nbag, int rows, int32_t* counts, int tid, int lane,
                                               bool& bad_id) {
  constexpr int kPer = kRun / W;
  int q = 0;  // this thread's bag, and where the next one starts
  int32_t nb = nbag > 1 ? off32[1] : INT32_MAX;
  const int b0 = tid * kRun;
  int32_t p0 = pa + b0 / W;  // the first position of this thread's run in chunk c
  for (int c = 0; c < nch; ++c, p0 += kChunk / W) {
    const bool got = mbar_wait(&full[slot], par, kWaitLimit);
    if (!__all_sync(0xffffffffu, got)) return false;
    const uint32_t bytes = c == nch - 1 ? last_bytes : (uint32_t)kChunk;
    if (count && (uint32_t)b0 < bytes) {  // chunk sizes are multiples of 16: a run is whole, half or absent
      const unsigned char* chunk = ring + slot * kChunk + b0;
      const uint4 v0 = *reinterpret_cast<const uint4*>(chunk);
      const uint4 v1 = (uint32_t)b0 + 16 < bytes ? *reinterpret_cast<const uint4*>(chunk + 16) : make_uint4(0, 0, 0, 0);
      const int n = (uint32_t)b0 + 16 < bytes ? kPer : kPer / 2;
      uint32_t id[kPer];  // an int64 id is in range only if its high word is 0
      if (W == 8) {
        id[0] = v0.y ? 0xffffffffu : v0.x;
        id[1] = v0.w ? 0xffffffffu : v0.z;
        id[2 % kPer] = v1.y ? 0xffffffffu : v1.x;
        id[3 % kPer] = v1.w ? 0xffffffffu : v1.z;
      } else {
        const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int k = 0; k < kPer; ++k) id[k] = u[k];
      }
      if (lut) {
        q = lut[p0 >> 5];
        nb = q < nbag - 1 ? off32[q + 1] : INT32_MAX;
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        if (k >= n) break;
        while (p0 + k >= nb) {
          ++q;
          nb = q < nbag - 1 ? off32[q + 1] : INT32_MAX;
        }
        if (id[k] < (uint32_t)rows) atomicAdd(&counts[q * kMaxK + (int)id[k]], 1);
        else bad_id = true;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == (uint32_t)R) {
      slot = 0;
      par ^= 1u;
    }
  }
  return true;
}

// One 16-byte piece of an id chunk, global -> shared, cached in L2 only.
__device__ __forceinline__ void cp_async16_cg(uint32_t dst, uintptr_t src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The producer warps: stream the id chunks of every unweighted tile of the
// CTA's range through the ring, running ahead of the consumers across tiles.
// Each producer thread copies its 16-byte pieces of a chunk and has the
// chunk's full barrier count its arrival once they have landed; a slot is
// refilled once all consumer warps have released it.  Every wait is bounded;
// on a timeout, or once the consumers stop, nothing more is issued, and no
// thread leaves before its copies have landed.
__device__ void produce_ids(const FwdArgs& a, const HistShape& h, int64_t tile_begin, int64_t tile_end, bool counts_only,
                            unsigned char* ring, uint64_t* full, uint64_t* empty, volatile int32_t* flags, int ptid) {
  const int w = a.indices.i32 ? 4 : 8;
  const int R = h.ring;
  const uint32_t ring_u32 = smem_u32(ring);
  uint32_t seq = 0, slot = 0, par = 0;  // chunks issued; slot and fill parity of the next
  for (int64_t tile = tile_begin; tile < tile_end && !flags[0]; ++tile) {
    const int t = (int)(tile / h.tpt);
    const int b0 = (int)(tile - (int64_t)t * h.tpt) * h.mb;
    const int nbag = min(h.mb, a.B - b0);
    if (!counts_only && a.psw != nullptr && __ldg(&a.meta[t].weighted)) continue;  // read directly
    const int64_t g0 = (int64_t)t * a.B + b0;
    const ChunkPlan cp(a.indices.p, w, a.offsets.ldg(g0), a.offsets.ldg(g0 + nbag), a.N);
    for (int c = 0; c < cp.nch; ++c, ++seq) {
      // a refill waits until all consumer warps released the slot's previous chunk
      if (seq >= (uint32_t)R && !mbar_wait(&empty[slot], par ^ 1u, kWaitLimit)) {
        report(a.status, TBE_DEV_TIMEOUT);
        flags[0] = 1;
      }
      if (flags[0]) break;
      const uint32_t bytes = cp.bytes(c);
      const uintptr_t src = cp.beg + (uintptr_t)c * kChunk;
      for (uint32_t j = (uint32_t)ptid * 16; j < bytes; j += kProducers * 16)
        cp_async16_cg(ring_u32 + slot * kChunk + j, src + j);
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&full[slot])) : "memory");
      if (++slot == (uint32_t)R) {
        slot = 0;
        par ^= 1u;
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename OutT, bool COUNTS_ONLY>
__global__ void __launch_bounds__(kThreads, 1) hist_kernel(const FwdArgs a, const HistShape h, int32_t* counts_out) {
  extern __shared__ unsigned char smem_raw[];
  const HistLayout L(h.maxD, h.b_esz, h.ring);
  // aligned by pointer arithmetic on the shared array itself, so that every
  // access through `base` stays a shared-memory access
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  int32_t* counts = reinterpret_cast<int32_t*>(base + L.counts);
  unsigned char* a32 = base + L.counts;  // the tf32 A tile spans the counts and 16-bit A regions
  unsigned char* a16 = base + L.a16;
  unsigned char* b_tile = base + L.b_tile;
  unsigned char* ring = base + L.ring;
  int64_t* off = reinterpret_cast<int64_t*>(base + L.off);
  uint32_t* over = reinterpret_cast<uint32_t*>(base + L.over);
  int32_t* off32 = reinterpret_cast<int32_t*>(base + L.over + (kM / 32) * 4);  // off - off[0] of a valid tile
  uint8_t* lut = reinterpret_cast<uint8_t*>(off32) + ((kM + 1) * 4 + 15) / 16 * 16;  // bag of position 32k
  uint64_t* mbar = reinterpret_cast<uint64_t*>(base + L.mbar);
  uint64_t* full = mbar + 1;
  uint64_t* empty = mbar + 1 + kRingMax;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.tmem);
  volatile int32_t* flags = reinterpret_cast<volatile int32_t*>(base + L.flags);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t ncols = h.maxD <= 32 ? 32 : (h.maxD <= 64 ? 64 : (h.maxD <= 128 ? 128 : 256));  // TMEM columns
  const int64_t ntiles = (int64_t)a.T * h.tpt;
  const int64_t TB = (int64_t)a.T * a.B;
  const int64_t tile_begin = ntiles * blockIdx.x / gridDim.x;
  const int64_t tile_end = ntiles * (blockIdx.x + 1) / gridDim.x;
  const int R = h.ring;

  if (tid == 0) {
    mbar_init(mbar);
    for (int k = 0; k < R; ++k) {
      mbar_init_count(&full[k], kProducers);
      mbar_init_count(&empty[k], kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    flags[0] = 0;
  }
  if (!COUNTS_ONLY && warp == 0) tmem_alloc(tmem_slot, ncols);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // the only barrier of all threads: from here the producer warp runs on its own
  if (tid >= kConsumers) {
    produce_ids(a, h, tile_begin, tile_end, COUNTS_ONLY, ring, full, empty, flags, tid - kConsumers);
    return;
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = COUNTS_ONLY ? 0u : *tmem_slot;
  float* stage = reinterpret_cast<float*>(base + L.stage) + warp * 32;
  uint32_t phase = 0;
  uint32_t slot = 0, par = 0;  // ring slot of the next chunk, and the parity of its fill
  bool stop = false;  // a bounded wait ran out: the consumers stop
  int cur_t = -1, cur_mode = -1;
  const int w = a.indices.i32 ? 4 : 8;

  for (int64_t tile = tile_begin; tile < tile_end; ++tile) {
    const int t = (int)(tile / h.tpt);
    const int b0 = (int)(tile - (int64_t)t * h.tpt) * h.mb;
    const int nbag = min(h.mb, a.B - b0);
    const TableMeta m = a.meta[t];
    const int rows = m.rows, D = m.D;
    const int K = (rows + 15) & ~15;  // MMA K, padded to 16
    const bool weighted = !COUNTS_ONLY && a.psw != nullptr && m.weighted;
    const int mode = weighted ? kModeTF32 : (m.dtype == TBE_F16 ? kModeF16 : kModeBF16);
    const int64_t g0 = (int64_t)t * a.B + b0;

    if (weighted) {
      for (int e = tid; e < K * (kM * 4 / 16); e += kConsumers) reinterpret_cast<int4*>(a32)[e] = make_int4(0, 0, 0, 0);
    } else {
      for (int e = tid; e < kM * kMaxK / 4; e += kConsumers) reinterpret_cast<int4*>(counts)[e] = make_int4(0, 0, 0, 0);
    }
    if (tid < kM / 32) over[tid] = 0;
    for (int q = tid; q <= nbag; q += kConsumers) off[q] = a.offsets.stream(g0 + q);
    if (!COUNTS_ONLY && (t != cur_t || mode != cur_mode)) {
      load_table(b_tile, a.weights + m.w_off, rows, K, D, m.dtype, mode, tid);
      cur_t = t;
      cur_mode = mode;
    }
    consumers_sync();
    // the chunks this tile streams (from the offsets as read, like the producer)
    const ChunkPlan cp(a.indices.p, w, off[0], off[nbag], a.N);
    bool bad = false;
    {
      // bag bounds: must start at 0, never decrease and end at N; a broken
      // tile is reported and pooled as empty (its chunks are still consumed)
      int b = off[0] < 0 || off[nbag] > a.N || (g0 == 0 && off[0] != 0) || (g0 + nbag == TB && off[nbag] != a.N);
      for (int q = tid; q < nbag; q += kConsumers) b |= off[q + 1] < off[q];
      bad = consumers_sync_or(b);
      if (bad) {
        if (tid == 0) report(a.status, TBE_DEV_BAD_OFFSETS);
        for (int q = tid; q <= nbag; q += kConsumers) off[q] = 0;
      } else {
        for (int q = tid; q <= nbag; q += kConsumers) off32[q] = (int32_t)(off[q] - off[0]);
      }
      consumers_sync();
      // lookup of every 32nd position's bag: entry k belongs to the bag whose
      // range holds position 32k; four threads share a bag's entries
      if (!bad && !weighted && off[nbag] - off[0] <= (int64_t)kLut * 32) {
        for (int i = tid; i < 4 * nbag; i += kConsumers) {
          const int q = i >> 2;
          for (int k = (off32[q] + 31) / 32 + (i & 3); k < (off32[q + 1] + 31) / 32; k += 4) lut[k] = (uint8_t)q;
        }
        consumers_sync();
      }
    }

    bool bad_id = false;
    if (!weighted) {
      // counts of every bag of the tile: the ragged ends read directly, the
      // aligned middle from the ring, where every thread counts its own run
      // of 32 bytes of each chunk and releases it (per warp) when done; its
      // positions only grow, so its bag index only moves forward
      if (!bad) {
        const int nh = (int)(cp.pa - cp.p0), nt = (int)(cp.p1 - cp.pe);
        if (tid < nh + nt) {
          const int64_t p = tid < nh ? cp.p0 + tid : cp.pe + (tid - nh);
          const uint64_t id = a.indices.id_bits(p);
          if (id < (uint64_t)rows) atomicAdd(&counts[tile_bag(off, nbag, p) * kMaxK + (int)id], 1);
          else bad_id = true;
        }
      }
      const int32_t pa = bad ? 0 : (int32_t)(cp.pa - off[0]);
      const uint8_t* tl = (off[nbag] - off[0] <= (int64_t)kLut * 32) ? lut : nullptr;  // else walk from run to run
      const uint32_t last = cp.nch > 0 ? cp.bytes(cp.nch - 1) : 0u;
      const bool ok = w == 8 ? consume_chunks<8>(ring, full, empty, R, slot, par, cp.nch, last, pa, !bad, off32, tl,
                                                 nbag, rows, counts, tid, lane, bad_id)
                             : consume_chunks<4>(ring, full, empty, R, slot, par, cp.nch, last, pa, !bad, off32, tl,
                                                 nbag, rows, counts, tid, lane, bad_id);
      if (!ok) stop = true;
      for (int b = tid; b < nbag; b += kConsumers)
        if (off[b + 1] - off[b] > (int64_t)kExactCount) atomicOr(&over[b >> 5], 1u << (b & 31));
    } else {
      // sums of per-sample weights: warp per bag, 32 lookups per step in
      // position order; lanes holding the same row are summed in lane order
      // by the lowest of them, which alone adds to the cell
      constexpr int kWU = 4;
      for (int q = warp; q < nbag; q += kWarps) {
        const int64_t s0 = off[q], e = off[q + 1];
        for (int64_t pb = s0; pb < e; pb += 32 * kWU) {
          uint64_t id[kWU];
          float wt[kWU];
#pragma unroll
          for (int u = 0; u < kWU; ++u) {
            const int64_t p = pb + u * 32 + lane;
            id[u] = p < e ? a.indices.id_bits(p) : ~0ull;
            wt[u] = p < e ? __ldg(a.psw + p) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < kWU; ++u) {
            if (pb + u * 32 >= e) break;  // warp-uniform
            const bool in = pb + u * 32 + lane < e;
            const bool ok = in && id[u] < (uint64_t)rows;
            bad_id |= in && !ok;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? id[u] : ~0ull);
            stage[lane] = wt[u];
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
    if (consumers_sync_or(stop)) {
      stop = true;
      break;
    }

    if (COUNTS_ONLY) {
      int32_t* dst = counts_out + m.row_base * (int64_t)a.B + (int64_t)b0 * rows;
      for (int e = tid; e < nbag * rows; e += kConsumers) {
        const int q = e / rows, r = e - q * rows;
        dst[e] = counts[q * kMaxK + r];
      }
      consumers_sync();
      continue;
    }

    // the A operand (see the header: one or two K passes per mode), one
    // 16-byte row of a core matrix per item (bag q = item mod 128, so the
    // 8 rows of a core matrix are written by neighbouring lanes)
    if (mode == kModeTF32) {
      for (int i = tid; i < kM * (K >> 2); i += kConsumers) {
        const int q = i & (kM - 1), k0 = (i >> 7) << 2;
        float4* cell = reinterpret_cast<float4*>(a32 + kmajor_byte(q, k0, kM, 4));
        const float4 c = *cell;
        const float4 s1 = make_float4(round_tf32(c.x), round_tf32(c.y), round_tf32(c.z), round_tf32(c.w));
        *cell = s1;
        *reinterpret_cast<float4*>(a32 + kmajor_byte(q, K + k0, kM, 4)) =
            make_float4(round_tf32(c.x - s1.x), round_tf32(c.y - s1.y), round_tf32(c.z - s1.z), round_tf32(c.w - s1.w));
      }
    } else {
      for (int i = tid; i < kM * (K >> 3); i += kConsumers) {
        const int q = i & (kM - 1), k0 = (i >> 7) << 3;
        const int4 c0 = *reinterpret_cast<const int4*>(&counts[q * kMaxK + k0]);
        const int4 c1 = *reinterpret_cast<const int4*>(&counts[q * kMaxK + k0 + 4]);
        const int32_t c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
          const int32_t x = min(c[k], (int32_t)kExactCount), y = min(c[k + 1], (int32_t)kExactCount);
          if (mode == kModeF16) {
            const __half2 h2 = __halves2half2(__int2half_rn(x), __int2half_rn(y));
            lo[k >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
            hi[k >> 1] = 0;
          } else {
            const __nv_bfloat162 l2 = __floats2bfloat162_rn((float)(x & 255), (float)(y & 255));
            const __nv_bfloat162 h2 = __floats2bfloat162_rn((float)(x - (x & 255)), (float)(y - (y & 255)));
            lo[k >> 1] = *reinterpret_cast<const uint32_t*>(&l2);
            hi[k >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
        *reinterpret_cast<uint4*>(a16 + kmajor_byte(q, k0, kM, 2)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (mode == kModeBF16)
          *reinterpret_cast<uint4*>(a16 + kmajor_byte(q, K + k0, kM, 2)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      }
    }
    // make the generic-proxy shared-memory writes visible to the tensor core
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    consumers_sync();
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
    if (consumers_sync_or(!ok)) {  // the consumers stop together
      if (tid == 0) report(a.status, TBE_DEV_TIMEOUT);
      stop = true;
      break;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    {
      // epilogue, 64 columns at a time through the 16-bit A region (free
      // once the MMA has read it): warps w and w+4 (w < 4) read the two
      // 32-column halves of TMEM lanes 32w.. (bag q = 32w + lane) into row q
      // of a [kM][64] fp32 staging tile, its 16-byte units XOR-swizzled by
      // q & 7 so that neither the row writes nor the row reads conflict;
      // then every warp stores whole bag rows, coalesced
      const int quarter = warp & 3, half = warp >> 2;
      const int q = quarter * 32 + lane;
      const bool is_over = q < nbag && ((over[q >> 5] >> (q & 31)) & 1u);
      float* stg = reinterpret_cast<float*>(a16);
      const bool vec = a.out_vec_ok;
      for (int c0 = 0; c0 < D; c0 += 64) {
        if (half < 2 && c0 + half * 32 < D) {  // warp-uniform
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(c0 + half * 32), v);
          if (is_over) {  // exact recount of an unweighted bag too long for 16-bit counts
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (c0 + half * 32 + c < D) {
                float acc = 0.f;
                for (int r = 0; r < rows; ++r) {
                  const uint16_t bits =
                      *reinterpret_cast<const uint16_t*>(b_tile + kmajor_byte(c0 + half * 32 + c, r, D, 2));
                  acc = __fadd_rn(acc, __fmul_rn((float)counts[q * kMaxK + r], table_value(bits, m.dtype)));
                }
                v[c] = acc;
              }
            }
          }
          if (a.mean && q < nbag) mean_scale(v, 32, off[q + 1] - off[q]);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(stg + q * 64 + (((half * 8 + j) ^ (q & 7)) << 2)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        consumers_sync();
        const int ncol = min(64, D - c0);
        if (2 * lane < ncol) {
          for (int r = warp; r < nbag; r += kWarps) {
            const float2 x = *reinterpret_cast<const float2*>(stg + r * 64 + (((lane >> 1) ^ (r & 7)) << 2) + ((lane & 1) << 1));
            OutT* dst = reinterpret_cast<OutT*>(a.out) + (int64_t)(b0 + r) * a.sumD + m.col_off + c0 + 2 * lane;
            store_pair<OutT>(dst, x.x, x.y, vec);
          }
        }
        consumers_sync();
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    consumers_sync();
  }
  if (stop && tid == 0) flags[0] = 1;  // a wait ran out: the producers issue nothing more
  if (!COUNTS_ONLY) {
    consumers_sync();
    if (warp == 0) tmem_dealloc(tmem, ncols);
  }
}

template <typename OutT, bool COUNTS_ONLY>
int launch_hist(const FwdArgs& a, HistShape h, int32_t* counts, cudaStream_t s) {
  auto kern = hist_kernel<OutT, COUNTS_ONLY>;
  // one CTA per SM (persistent); the id ring takes what shared memory is left
  int dev = 0, smem_max = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return TBE_ERR_CUDA;
  const size_t fixed = (size_t)HistLayout(h.maxD, h.b_esz, 0).total + 1024;  // + alignment slack
  if ((size_t)smem_max < fixed + (size_t)kRingMin * kChunk) return TBE_ERR_UNSUPPORTED;
  h.ring = (int)std::min<size_t>(kRingMax, ((size_t)smem_max - fixed) / kChunk);
  const size_t smem = fixed + (size_t)h.ring * kChunk;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess)
    return TBE_ERR_CUDA;
  const int64_t ntiles = (int64_t)a.T * h.tpt;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ntiles, (int64_t)sm_count()));
  kern<<<grid, kThreads, smem, s>>>(a, h, counts);
  return check_launch();
}

}  // namespace

int launch_forward_histogram(const Plan& p, const FwdArgs& a, int32_t* counts_out, cudaStream_t s) {
  HistShape h;
  h.maxD = p.maxD;
  h.b_esz = (!counts_out && a.psw != nullptr && p.any_weighted) ? 4 : 2;
  // bags per tile: at most kM, and as few as make the tiles a whole number
  // of waves of one CTA per SM, so that every CTA counts about as many ids
  const int64_t waves = std::max<int64_t>(1, ((int64_t)p.T * ((a.B + kM - 1) / kM) + sm_count() - 1) / sm_count());
  const int64_t per_table = std::max<int64_t>(1, (waves * sm_count() + p.T - 1) / p.T);
  h.mb = (int)std::min<int64_t>(kM, std::max<int64_t>(1, (a.B + per_table - 1) / per_table));
  h.tpt = (a.B + h.mb - 1) / h.mb;
  h.ring = kRingMin;
  if (counts_out) return launch_hist<float, true>(a, h, counts_out, s);
  switch (p.out_dtype) {
    case TBE_F32: return launch_hist<float, false>(a, h, nullptr, s);
    case TBE_F16: return launch_hist<__half, false>(a, h, nullptr, s);
    default: return launch_hist<__nv_bfloat16, false>(a, h, nullptr, s);
  }
}

}  // namespace tbe
