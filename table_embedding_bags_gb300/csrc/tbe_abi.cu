// tbe_abi.cu -- the C ABI of libtbe: argument validation, plans, dispatch,
// tuning and stage tracing.  Every entry point only enqueues kernels on the
// caller's stream; none synchronises or allocates device memory.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tbe_internal.cuh"

namespace tbe {

// Defaults, from sweeps timed on GB300 with `bench.py --sweep`:
//  - long_run_threshold 32 with the automatic chunk (64 for batches of about
//    0.3-1.3 M lookups, 256 from about 5 M) was the fastest, or within 3 %
//    of it, of threshold {16, 32, 64, 128, 256} x chunk {64, 128, 256} on the
//    mid-size, backward-skew and three run-length band workloads; a threshold
//    of 256 was 1.34x slower on runs of 32..255 lookups;
//  - hist_min_mean_bag 0 selects the measured gate: the histogram path beat
//    the gather path from a mean bag length of 16 on fp16 and bf16 tables of
//    8..64 rows, one or four tables (D = 128), and with per-sample weights
//    from 16 on 16-row tables but only from 32 on 64-row tables.
static Tuning g_tuning = {/*long_run_threshold=*/32, /*long_chunk=*/0, /*fwd_unroll=*/4,
                          /*fwd_blocks_per_sm=*/0, /*hist_min_mean_bag=*/0,
                          /*short_item_lookups=*/32, /*fwd_lanes_per_row=*/16,
                          /*red_unroll=*/4, /*fwd_ring=*/3};

const Tuning& tuning() { return g_tuning; }

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

int check_launch() { return cudaGetLastError() == cudaSuccess ? TBE_OK : TBE_ERR_CUDA; }

// ---------------------------------------------------------------------------
// bounded-wait self-test
// ---------------------------------------------------------------------------
namespace {
// A look-back word that no kernel ever publishes (device memory is zero at
// load time and nothing writes it).
__device__ uint32_t g_unpublished_word;

// One thread runs one of the library's bounded waits on something that
// never completes -- kind 0: the look-back word wait of the backward's scans,
// kind 1: the mbarrier wait of the histogram path (a barrier that expects
// one arrival; nothing arrives and no copy is in flight) -- and reports
// TBE_DEV_TIMEOUT when it gives up after `polls` polls.
__global__ void wait_selftest_kernel(int32_t kind, int32_t polls, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  bool ok;
  if (kind == 0) {
    ok = poll_word(&g_unpublished_word, 0xffffffffu, polls) != 0;
  } else {
    mbar_init(&bar);
    ok = mbar_wait(&bar, 0, polls);
  }
  if (!ok) report(status, TBE_DEV_TIMEOUT);
}
}  // namespace

// ---------------------------------------------------------------------------
// stage tracing
// ---------------------------------------------------------------------------
namespace {
constexpr int kMaxStages = 32;
struct Trace {
  std::mutex mu;
  bool on = false;
  int device = -1;
  cudaEvent_t ev[kMaxStages + 1] = {};
  const char* names[kMaxStages + 1] = {};
  int n = 0;  // events recorded by the last call (including the start event)
};
Trace g_trace;
}  // namespace

// Records `ev` on `s`; inside a stream capture the record becomes a graph
// node (external record), so replays of the graph time the same stages.
static cudaError_t record(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  return cudaEventRecord(ev, s);
}

void trace_begin(cudaStream_t s) {
  if (!g_trace.on) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  g_trace.n = 0;
  if (record(g_trace.ev[0], s) == cudaSuccess) g_trace.n = 1;
  g_trace.names[0] = "start";
}

void trace_mark(cudaStream_t s, const char* name) {
  if (!g_trace.on) return;
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (g_trace.n == 0 || g_trace.n > kMaxStages) return;
  if (record(g_trace.ev[g_trace.n], s) == cudaSuccess) g_trace.names[g_trace.n++] = name;
}

}  // namespace tbe

using namespace tbe;

struct tbe_plan : public tbe::Plan {};

extern "C" {

const char* tbe_version(void) { return "libtbe 0.1 (sm_103a)"; }

int tbe_wait_selftest(int32_t kind, int32_t polls, int32_t* dev_status, void* stream) {
  if ((kind != 0 && kind != 1) || polls < 1 || polls > (1 << 20) || !dev_status) return TBE_ERR_INVALID_ARG;
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(kind, polls, dev_status);
  return check_launch();
}

const char* tbe_status_string(int32_t code) {
  switch (code) {
    case TBE_OK: return "ok";
    case TBE_ERR_INVALID_ARG: return "invalid argument";
    case TBE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case TBE_ERR_CUDA: return "CUDA error";
    case TBE_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int tbe_get_tuning(tbe_tuning* out) {
  if (!out) return TBE_ERR_INVALID_ARG;
  out->long_run_threshold = g_tuning.long_run_threshold;
  out->long_chunk = g_tuning.long_chunk;
  out->fwd_unroll = g_tuning.fwd_unroll;
  out->fwd_blocks_per_sm = g_tuning.fwd_blocks_per_sm;
  out->hist_min_mean_bag = g_tuning.hist_min_mean_bag;
  out->short_item_lookups = g_tuning.short_item_lookups;
  out->fwd_lanes_per_row = g_tuning.fwd_lanes_per_row;
  out->red_unroll = g_tuning.red_unroll;
  out->fwd_ring = g_tuning.fwd_ring;
  return TBE_OK;
}

int tbe_set_tuning(const tbe_tuning* in) {
  if (!in) return TBE_ERR_INVALID_ARG;
  if (in->long_run_threshold < 1 || in->long_run_threshold > (1 << 20)) return TBE_ERR_INVALID_ARG;
  if (in->long_chunk != 0 && (in->long_chunk < 32 || in->long_chunk > 65536 || (in->long_chunk % 32) != 0))
    return TBE_ERR_INVALID_ARG;
  if (in->fwd_unroll != 4 && in->fwd_unroll != 8) return TBE_ERR_INVALID_ARG;
  if (in->fwd_lanes_per_row < 1 || in->fwd_lanes_per_row > 32 ||
      (in->fwd_lanes_per_row & (in->fwd_lanes_per_row - 1)) != 0)
    return TBE_ERR_INVALID_ARG;
  if (in->fwd_blocks_per_sm < 0 || in->fwd_blocks_per_sm > 32) return TBE_ERR_INVALID_ARG;
  if (in->hist_min_mean_bag < 0) return TBE_ERR_INVALID_ARG;
  if (in->red_unroll != 4 && in->red_unroll != 8) return TBE_ERR_INVALID_ARG;
  if (in->fwd_ring < 0 || in->fwd_ring > 3) return TBE_ERR_INVALID_ARG;
  if (in->short_item_lookups < 32 || in->short_item_lookups > (1 << 20)) return TBE_ERR_INVALID_ARG;
  g_tuning.long_run_threshold = in->long_run_threshold;
  g_tuning.long_chunk = in->long_chunk;
  g_tuning.fwd_unroll = in->fwd_unroll;
  g_tuning.fwd_blocks_per_sm = in->fwd_blocks_per_sm;
  g_tuning.hist_min_mean_bag = in->hist_min_mean_bag;
  g_tuning.short_item_lookups = in->short_item_lookups;
  g_tuning.fwd_lanes_per_row = in->fwd_lanes_per_row;
  g_tuning.red_unroll = in->red_unroll;
  g_tuning.fwd_ring = in->fwd_ring;
  return TBE_OK;
}

int tbe_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TBE_ERR_CUDA;
  if (on && (g_trace.device != dev || g_trace.ev[0] == nullptr)) {
    for (int k = 0; k <= kMaxStages; ++k) {
      if (g_trace.ev[k]) cudaEventDestroy(g_trace.ev[k]);
      if (cudaEventCreate(&g_trace.ev[k]) != cudaSuccess) return TBE_ERR_CUDA;
    }
    g_trace.device = dev;
  }
  g_trace.on = on != 0;
  g_trace.n = 0;
  return TBE_OK;
}

int tbe_trace_read(float* stage_ms, const char** stage_names, int32_t max_stages) {
  std::lock_guard<std::mutex> lk(g_trace.mu);
  if (g_trace.n < 1) return 0;
  if (cudaEventSynchronize(g_trace.ev[g_trace.n - 1]) != cudaSuccess) return -TBE_ERR_CUDA;
  int ns = std::min<int>(g_trace.n - 1, max_stages);
  for (int k = 0; k < ns; ++k) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_trace.ev[k], g_trace.ev[k + 1]) != cudaSuccess) return -TBE_ERR_CUDA;
    if (stage_ms) stage_ms[k] = ms;
    if (stage_names) stage_names[k] = g_trace.names[k + 1];
  }
  return ns;
}

// ---------------------------------------------------------------------------
// plans
// ---------------------------------------------------------------------------

size_t tbe_plan_device_bytes(int32_t T) {
  if (T < 1 || T > TBE_MAX_TABLES) return 0;
  size_t b = sizeof(TableMeta) * (size_t)(T + 1);
  return (b + 255) / 256 * 256;
}

static int elem_size(int32_t dt) { return dt == TBE_F32 ? 4 : 2; }

int tbe_plan_create(const tbe_layout* L, void* dev_meta, size_t dev_meta_bytes, void* stream,
                    tbe_plan** plan_out) {
  if (!L || !plan_out || !dev_meta) return TBE_ERR_INVALID_ARG;
  *plan_out = nullptr;
  const int32_t T = L->T;
  if (T < 1 || T > TBE_MAX_TABLES) return TBE_ERR_INVALID_ARG;
  if (!L->table_row_base || !L->D_offsets || !L->weights_offsets || !L->weights_dtype)
    return TBE_ERR_INVALID_ARG;
  if (L->out_dtype < TBE_F32 || L->out_dtype > TBE_BF16) return TBE_ERR_INVALID_ARG;
  if (L->pooling != TBE_POOL_SUM && L->pooling != TBE_POOL_MEAN) return TBE_ERR_INVALID_ARG;
  if (dev_meta_bytes < tbe_plan_device_bytes(T) || ((uintptr_t)dev_meta & 15)) return TBE_ERR_INVALID_ARG;
  if (L->table_row_base[0] != 0 || L->D_offsets[0] != 0) return TBE_ERR_INVALID_ARG;

  tbe_plan* p = new (std::nothrow) tbe_plan();
  if (!p) return TBE_ERR_INVALID_ARG;
  p->hmeta = new (std::nothrow) TableMeta[T + 1];
  if (!p->hmeta) { delete p; return TBE_ERR_INVALID_ARG; }
  std::memset(p->hmeta, 0, sizeof(TableMeta) * (T + 1));
  int status = TBE_OK;
  int dtype_mask = 0, any_weighted = 0, maxD = 0;
  const int osz = elem_size(L->out_dtype);
  int out_vec_ok = 1;
  for (int32_t t = 0; t < T && status == TBE_OK; ++t) {
    const int64_t rows = L->table_row_base[t + 1] - L->table_row_base[t];
    const int32_t D = L->D_offsets[t + 1] - L->D_offsets[t];
    const int32_t dt = L->weights_dtype[t];
    if (rows < 0 || D <= 0 || dt < TBE_F32 || dt > TBE_BF16 || L->weights_offsets[t] < 0) {
      status = TBE_ERR_INVALID_ARG;
      break;
    }
    if (rows >= (int64_t(1) << 31) || ((int64_t)D * elem_size(dt)) % 16 != 0 ||
        (L->weights_offsets[t] % 16) != 0) {
      status = TBE_ERR_UNSUPPORTED;
      break;
    }
    TableMeta& m = p->hmeta[t];
    m.w_off = L->weights_offsets[t];
    m.row_base = L->table_row_base[t];
    m.rows = (int32_t)rows;
    m.col_off = L->D_offsets[t];
    m.D = D;
    m.dtype = (uint8_t)dt;
    m.weighted = L->table_weighted ? (L->table_weighted[t] ? 1 : 0) : 1;
    dtype_mask |= 1 << dt;
    any_weighted |= m.weighted;
    maxD = std::max(maxD, D);
    if (((int64_t)m.col_off * osz) % 16 != 0) out_vec_ok = 0;
  }
  const int64_t total_rows = L->table_row_base[T];
  if (status == TBE_OK && (total_rows >= 0xffffffffLL || (int64_t)L->D_offsets[T] >= (int64_t(1) << 31)))
    status = TBE_ERR_UNSUPPORTED;
  if (status != TBE_OK) {
    delete[] p->hmeta;
    delete p;
    return status;
  }
  p->hmeta[T].row_base = total_rows;
  p->T = T;
  p->out_dtype = L->out_dtype;
  p->pooling = L->pooling;
  p->sumD = L->D_offsets[T];
  p->maxD = maxD;
  p->total_rows = total_rows;
  int kb = 1;
  while (kb < 32 && (total_rows >> kb) != 0) ++kb;
  p->key_bits = kb;
  int64_t max_rows = 0;
  for (int32_t t = 0; t < T; ++t) max_rows = std::max<int64_t>(max_rows, p->hmeta[t].rows);
  int sb = 1;
  while (sb < 32 && (max_rows >> sb) != 0) ++sb;
  p->seg_bits = sb;
  p->dtype_mask = dtype_mask;
  p->any_weighted = any_weighted;
  if (((int64_t)p->sumD * osz) % 16 != 0) out_vec_ok = 0;
  p->out_vec_ok = out_vec_ok;
  p->max_row_bytes = 0;
  for (int32_t t = 0; t < T; ++t)
    p->max_row_bytes = std::max(p->max_row_bytes, p->hmeta[t].D * elem_size(p->hmeta[t].dtype));
  p->uniform = 1;
  for (int32_t t = 1; t < T; ++t)
    if (p->hmeta[t].D != p->hmeta[0].D || p->hmeta[t].dtype != p->hmeta[0].dtype ||
        p->hmeta[t].weighted != p->hmeta[0].weighted)
      p->uniform = 0;
  // histogram path: every table small enough for one MMA tile, fp16 or bf16
  p->hist_ok = T >= 1;
  for (int32_t t = 0; t < T; ++t) {
    const TableMeta& m = p->hmeta[t];
    if (!(m.dtype == TBE_F16 || m.dtype == TBE_BF16) || m.rows < 1 || m.rows > TBE_HIST_MAX_ROWS ||
        m.D % 16 != 0 || m.D > 256)
      p->hist_ok = 0;
  }
  cudaGetDevice(&p->device);
  p->dmeta = reinterpret_cast<const TableMeta*>(dev_meta);
  if (cudaMemcpyAsync(dev_meta, p->hmeta, sizeof(TableMeta) * (T + 1), cudaMemcpyHostToDevice,
                      (cudaStream_t)stream) != cudaSuccess) {
    delete[] p->hmeta;
    delete p;
    return TBE_ERR_CUDA;
  }
  *plan_out = p;
  return TBE_OK;
}

void tbe_plan_destroy(tbe_plan* plan) {
  if (!plan) return;
  delete[] plan->hmeta;
  delete plan;
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

static int check_common(const tbe_plan* plan, const void* indices, int64_t N, const void* offsets, int32_t B) {
  if (!plan) return TBE_ERR_INVALID_ARG;
  if (B < 0 || N < 0 || N >= (int64_t(1) << 30)) return TBE_ERR_INVALID_ARG;
  if ((int64_t)plan->T * B >= (int64_t(1) << 31)) return TBE_ERR_UNSUPPORTED;
  if ((int64_t)plan->T * B > 0 && !offsets) return TBE_ERR_INVALID_ARG;
  if ((int64_t)plan->T * B == 0 && N != 0) return TBE_ERR_INVALID_ARG;  // no bag can hold a lookup
  if (N > 0 && !indices) return TBE_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TBE_ERR_CUDA;
  if (dev != plan->device) return TBE_ERR_INVALID_ARG;
  return TBE_OK;
}

// Mean bag length from which TBE_PATH_AUTO takes the histogram path.
static int64_t hist_gate(const tbe_plan& plan, const float* psw) {
  if (g_tuning.hist_min_mean_bag > 0) return g_tuning.hist_min_mean_bag;
  return psw != nullptr && plan.any_weighted ? 32 : 16;
}

static bool hist_eligible(const tbe_plan* plan) { return plan->hist_ok; }

// Shared by the int64 and int32 forward entry points.
static int forward_call(const tbe_plan* plan, const void* weights, IdxPtr indices, int64_t N, IdxPtr offsets,
                        int32_t B, const float* per_sample_weights, void* out, int32_t* dev_status, void* stream,
                        int32_t path) {
  int st = check_common(plan, indices.p, N, offsets.p, B);
  if (st != TBE_OK) return st;
  if (path < TBE_PATH_AUTO || path > TBE_PATH_HISTOGRAM) return TBE_ERR_INVALID_ARG;
  if ((int64_t)plan->T * B == 0) return TBE_OK;
  if (!out || !weights) return TBE_ERR_INVALID_ARG;
  if ((uintptr_t)weights & 15) return TBE_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  FwdArgs a;
  a.weights = reinterpret_cast<const uint8_t*>(weights);
  a.meta = plan->dmeta;
  a.indices = indices;
  a.offsets = offsets;
  a.psw = per_sample_weights;
  a.out = out;
  a.status = dev_status;
  a.T = plan->T;
  a.B = B;
  a.N = N;
  a.sumD = plan->sumD;
  a.out_vec_ok = plan->out_vec_ok && (((uintptr_t)out & 15) == 0);
  a.lpr_max = g_tuning.fwd_lanes_per_row;
  a.balance = plan->uniform ? 0 : 1;
  a.mean = plan->pooling == TBE_POOL_MEAN;
  a.split = 0;  // chosen by the stream kernel's launch
  bool hist = false;
  if (path == TBE_PATH_HISTOGRAM) {
    if (!hist_eligible(plan)) return TBE_ERR_UNSUPPORTED;
    hist = true;
  } else if (path == TBE_PATH_AUTO) {
    hist = hist_eligible(plan) && N >= hist_gate(*plan, per_sample_weights) * (int64_t)plan->T * B;
  }
  trace_begin(s);
  st = hist ? launch_forward_histogram(*plan, a, nullptr, s) : launch_forward_gather(*plan, a, s);
  trace_mark(s, hist ? "fwd_histogram" : "fwd_gather");
  return st;
}

int tbe_forward_path(const tbe_plan* plan, const void* weights, const int64_t* indices, int64_t N,
                     const int64_t* offsets, int32_t B, const float* per_sample_weights, void* out,
                     int32_t* dev_status, void* stream, int32_t path) {
  return forward_call(plan, weights, IdxPtr{indices, 0}, N, IdxPtr{offsets, 0}, B, per_sample_weights, out,
                      dev_status, stream, path);
}

int tbe_forward_i32(const tbe_plan* plan, const void* weights, const int32_t* indices, int64_t N,
                    const int32_t* offsets, int32_t B, const float* per_sample_weights, void* out,
                    int32_t* dev_status, void* stream, int32_t path) {
  return forward_call(plan, weights, IdxPtr{indices, 1}, N, IdxPtr{offsets, 1}, B, per_sample_weights, out,
                      dev_status, stream, path);
}

int tbe_forward(const tbe_plan* plan, const void* weights, const int64_t* indices, int64_t N,
                const int64_t* offsets, int32_t B, const float* per_sample_weights, void* out,
                int32_t* dev_status, void* stream) {
  return tbe_forward_path(plan, weights, indices, N, offsets, B, per_sample_weights, out, dev_status,
                          stream, TBE_PATH_AUTO);
}

int tbe_histogram_counts(const tbe_plan* plan, const int64_t* indices, int64_t N, const int64_t* offsets,
                         int32_t B, int32_t* counts, int32_t* dev_status, void* stream) {
  int st = check_common(plan, indices, N, offsets, B);
  if (st != TBE_OK) return st;
  if (!plan->hist_ok) return TBE_ERR_UNSUPPORTED;
  if (B == 0) return TBE_OK;
  if (!counts) return TBE_ERR_INVALID_ARG;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.meta = plan->dmeta;
  a.indices = IdxPtr{indices, 0};
  a.offsets = IdxPtr{offsets, 0};
  a.status = dev_status;
  a.T = plan->T;
  a.B = B;
  a.N = N;
  a.sumD = plan->sumD;
  return launch_forward_histogram(*plan, a, counts, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------

size_t tbe_backward_workspace_bytes(const tbe_plan* plan, int32_t B, int64_t N) {
  if (!plan || B < 0 || N < 0) return 0;
  return backward_workspace_bytes(*plan, B, N);
}

// Shared by tbe_backward and tbe_backward_update: checks and launches the
// backward; `opt` (may be null) fuses the exact optimizer into the reducer.
// stages: kBwdIndex and/or kBwdReduce (tbe_backward runs both; the index
// stages read no grad_out, the reduction no ids or offsets).
static int backward_call(const tbe_plan* plan, const float* grad_out, IdxPtr indices, int64_t N,
                         IdxPtr offsets, int32_t B, const float* per_sample_weights, int64_t* unique_rows,
                         int32_t* run_starts, int32_t* sorted_positions, float* row_grads,
                         int64_t row_grads_capacity, int64_t* unique_count, void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, void* stream, const tbe_optimizer* opt, void* weights,
                         float* momentum, int stages = kBwdIndex | kBwdReduce) {
  const bool index = stages & kBwdIndex, reduce = stages & kBwdReduce;
  // the reduction alone reads no ids or offsets: check the rest as for a full call
  int st = check_common(plan, index ? indices.p : (const void*)plan, N, index ? offsets.p : (const void*)plan, B);
  if (st != TBE_OK) return st;
  if (!unique_count || row_grads_capacity < 0) return TBE_ERR_INVALID_ARG;
  if (N > 0 && !unique_rows) return TBE_ERR_INVALID_ARG;
  if (N > 0 && reduce && (!grad_out || (!opt && !row_grads && row_grads_capacity > 0))) return TBE_ERR_INVALID_ARG;
  if ((uintptr_t)grad_out & 15) return TBE_ERR_UNSUPPORTED;
  if ((plan->sumD % 4) != 0) return TBE_ERR_UNSUPPORTED;
  for (int t = 0; t < plan->T; ++t)
    if (plan->hmeta[t].D % 4 != 0) return TBE_ERR_UNSUPPORTED;
  const size_t need = backward_workspace_bytes(*plan, B, N);
  if (workspace_bytes < need || (need > 0 && !workspace)) return TBE_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255) != 0) return TBE_ERR_INVALID_ARG;
  BwdArgs a;
  a.grad_out = grad_out;
  a.meta = plan->dmeta;
  a.indices = indices;
  a.offsets = offsets;
  a.psw = per_sample_weights;
  a.unique_rows = unique_rows;
  a.run_starts = run_starts;
  a.sorted_positions = sorted_positions;
  a.row_grads = opt ? nullptr : row_grads;
  a.row_grads_capacity = opt ? INT64_MAX : row_grads_capacity;
  a.unique_count = unique_count;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.status = dev_status;
  a.T = plan->T;
  a.B = B;
  a.N = N;
  a.sumD = plan->sumD;
  a.opt_kind = opt ? opt->kind : -1;
  a.lr = opt ? opt->learning_rate : 0.f;
  a.eps = opt ? opt->eps : 0.f;
  a.weights = static_cast<uint8_t*>(weights);
  a.momentum = momentum;
  cudaStream_t s = (cudaStream_t)stream;
  trace_begin(s);
  return launch_backward(*plan, a, s, stages);
}

int tbe_backward(const tbe_plan* plan, const float* grad_out, const int64_t* indices, int64_t N,
                 const int64_t* offsets, int32_t B, const float* per_sample_weights,
                 int64_t* unique_rows, int32_t* run_starts, int32_t* sorted_positions, float* row_grads,
                 int64_t row_grads_capacity, int64_t* unique_count, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return backward_call(plan, grad_out, IdxPtr{indices, 0}, N, IdxPtr{offsets, 0}, B, per_sample_weights,
                       unique_rows, run_starts, sorted_positions, row_grads, row_grads_capacity, unique_count,
                       workspace, workspace_bytes, dev_status, stream, nullptr, nullptr, nullptr);
}

int tbe_backward_i32(const tbe_plan* plan, const float* grad_out, const int32_t* indices, int64_t N,
                     const int32_t* offsets, int32_t B, const float* per_sample_weights, int64_t* unique_rows,
                     int32_t* run_starts, int32_t* sorted_positions, float* row_grads, int64_t row_grads_capacity,
                     int64_t* unique_count, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream) {
  return backward_call(plan, grad_out, IdxPtr{indices, 1}, N, IdxPtr{offsets, 1}, B, per_sample_weights,
                       unique_rows, run_starts, sorted_positions, row_grads, row_grads_capacity, unique_count,
                       workspace, workspace_bytes, dev_status, stream, nullptr, nullptr, nullptr);
}

// Optimizer arguments valid on the host (kind, finite rate, eps >= 0).
static bool opt_ok(const tbe_optimizer* opt) {
  return opt && (opt->kind == TBE_OPT_EXACT_SGD || opt->kind == TBE_OPT_EXACT_ROWWISE_ADAGRAD) &&
         std::isfinite(opt->learning_rate) && std::isfinite(opt->eps) && opt->eps >= 0.f;
}

// Shared by the int64 and int32 fused entry points.
static int backward_update_call(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                                const float* grad_out, IdxPtr indices, int64_t N, IdxPtr offsets, int32_t B,
                                const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                                int32_t* sorted_positions, int64_t* unique_count, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!plan || !opt_ok(opt)) return TBE_ERR_INVALID_ARG;
  if (plan->maxD > 128) return TBE_ERR_UNSUPPORTED;  // a row gradient is one quad per lane of one warp
  if (N > 0 && (!weights || (opt->kind == TBE_OPT_EXACT_ROWWISE_ADAGRAD && !momentum))) return TBE_ERR_INVALID_ARG;
  if ((uintptr_t)weights & 15) return TBE_ERR_UNSUPPORTED;
  return backward_call(plan, grad_out, indices, N, offsets, B, per_sample_weights, unique_rows, run_starts,
                       sorted_positions, nullptr, 0, unique_count, workspace, workspace_bytes, dev_status, stream,
                       opt, weights, momentum);
}

int tbe_backward_update(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                        const float* grad_out, const int64_t* indices, int64_t N, const int64_t* offsets,
                        int32_t B, const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                        int32_t* sorted_positions, int64_t* unique_count, void* workspace,
                        size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return backward_update_call(plan, opt, weights, momentum, grad_out, IdxPtr{indices, 0}, N, IdxPtr{offsets, 0}, B,
                              per_sample_weights, unique_rows, run_starts, sorted_positions, unique_count,
                              workspace, workspace_bytes, dev_status, stream);
}

int tbe_backward_update_i32(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                            const float* grad_out, const int32_t* indices, int64_t N, const int32_t* offsets,
                            int32_t B, const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                            int32_t* sorted_positions, int64_t* unique_count, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return backward_update_call(plan, opt, weights, momentum, grad_out, IdxPtr{indices, 1}, N, IdxPtr{offsets, 1}, B,
                              per_sample_weights, unique_rows, run_starts, sorted_positions, unique_count,
                              workspace, workspace_bytes, dev_status, stream);
}

int tbe_backward_index(const tbe_plan* plan, const int64_t* indices, int64_t N, const int64_t* offsets, int32_t B,
                       const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                       int32_t* sorted_positions, int64_t row_grads_capacity, int64_t* unique_count, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return backward_call(plan, nullptr, IdxPtr{indices, 0}, N, IdxPtr{offsets, 0}, B, per_sample_weights, unique_rows,
                       run_starts, sorted_positions, nullptr, row_grads_capacity, unique_count, workspace,
                       workspace_bytes, dev_status, stream, nullptr, nullptr, nullptr, kBwdIndex);
}

int tbe_backward_index_i32(const tbe_plan* plan, const int32_t* indices, int64_t N, const int32_t* offsets,
                           int32_t B, const float* per_sample_weights, int64_t* unique_rows, int32_t* run_starts,
                           int32_t* sorted_positions, int64_t row_grads_capacity, int64_t* unique_count,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return backward_call(plan, nullptr, IdxPtr{indices, 1}, N, IdxPtr{offsets, 1}, B, per_sample_weights, unique_rows,
                       run_starts, sorted_positions, nullptr, row_grads_capacity, unique_count, workspace,
                       workspace_bytes, dev_status, stream, nullptr, nullptr, nullptr, kBwdIndex);
}

int tbe_backward_reduce(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                        const float* grad_out, int64_t N, int32_t B, const float* per_sample_weights,
                        int64_t* unique_rows, int32_t* run_starts, float* row_grads, int64_t row_grads_capacity,
                        int64_t* unique_count, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream) {
  if (opt) {
    if (!plan || !opt_ok(opt)) return TBE_ERR_INVALID_ARG;
    if (plan->maxD > 128) return TBE_ERR_UNSUPPORTED;  // a row gradient is one quad per lane of one warp
    if (N > 0 && (!weights || (opt->kind == TBE_OPT_EXACT_ROWWISE_ADAGRAD && !momentum))) return TBE_ERR_INVALID_ARG;
    if ((uintptr_t)weights & 15) return TBE_ERR_UNSUPPORTED;
  }
  return backward_call(plan, grad_out, IdxPtr{nullptr, 0}, N, IdxPtr{nullptr, 0}, B, per_sample_weights, unique_rows,
                       run_starts, nullptr, row_grads, row_grads_capacity, unique_count, workspace, workspace_bytes,
                       dev_status, stream, opt, weights, momentum, kBwdReduce);
}

int tbe_exact_update(const tbe_plan* plan, const tbe_optimizer* opt, void* weights, float* momentum,
                     const int64_t* unique_rows, int64_t max_unique, const float* row_grads,
                     int64_t row_grads_capacity, const int64_t* unique_count, int32_t* dev_status,
                     void* stream) {
  if (!plan || !opt || max_unique < 0 || row_grads_capacity < 0) return TBE_ERR_INVALID_ARG;
  if (opt->kind != TBE_OPT_EXACT_SGD && opt->kind != TBE_OPT_EXACT_ROWWISE_ADAGRAD) return TBE_ERR_INVALID_ARG;
  if (!std::isfinite(opt->learning_rate) || !std::isfinite(opt->eps) || opt->eps < 0.f)
    return TBE_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TBE_ERR_CUDA;
  if (dev != plan->device) return TBE_ERR_INVALID_ARG;
  if (!unique_count) return TBE_ERR_INVALID_ARG;
  if (max_unique > 0 && (!weights || !unique_rows || (!row_grads && row_grads_capacity > 0)))
    return TBE_ERR_INVALID_ARG;
  if (max_unique > 0 && opt->kind == TBE_OPT_EXACT_ROWWISE_ADAGRAD && !momentum) return TBE_ERR_INVALID_ARG;
  if (((uintptr_t)row_grads & 15) || ((uintptr_t)weights & 15)) return TBE_ERR_UNSUPPORTED;
  for (int t = 0; t < plan->T; ++t)
    if (plan->hmeta[t].D % 4 != 0) return TBE_ERR_UNSUPPORTED;
  UpdArgs a;
  a.weights = static_cast<uint8_t*>(weights);
  a.meta = plan->dmeta;
  a.momentum = momentum;
  a.unique_rows = unique_rows;
  a.row_grads = row_grads;
  a.unique_count = unique_count;
  a.max_unique = max_unique;
  a.row_grads_capacity = row_grads_capacity;
  a.status = dev_status;
  a.T = plan->T;
  a.kind = opt->kind;
  a.lr = opt->learning_rate;
  a.eps = opt->eps;
  cudaStream_t s = (cudaStream_t)stream;
  trace_begin(s);
  return launch_exact_update(*plan, a, s);
}

}  // extern "C"
