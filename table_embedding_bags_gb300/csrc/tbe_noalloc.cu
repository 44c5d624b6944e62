// tbe_noalloc.cu -- the backward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the
// backward: a plugin inside a serving or training engine is handed a stream
// and the tensors it reads and writes, while the engine owns every other
// byte of device memory (allocating behind its back breaks its memory budget,
// and cudaMalloc may synchronise the device in the middle of its pipeline).
// For them this file provides
// tbe_backward_static_workspace(): the same computation as tbe_backward(),
// whose scratch space is one fixed array compiled into the library instead of
// a caller-provided workspace.  The caller still passes every input and output.
//
// The array lives in every GPU that loads the library until the process
// exits.  Its device address is looked up once per device, on the first call
// made with that device current.  All calls on a device share the one array:
// the backward clears the parts that must start at zero itself, but two calls
// whose work overlaps on the GPU (on different streams) race on it and must
// be serialised by the caller.
#include <mutex>

#include "tbe_internal.cuh"

// file-scope scratch of the static-workspace backward (see the header)
static __device__ __align__(256) unsigned char g_tbe_static_workspace[TBE_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_workspace_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per device).
int static_workspace(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TBE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_workspace_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tbe_static_workspace) != cudaSuccess || p == nullptr) return TBE_ERR_CUDA;
    g_workspace_addr[dev] = p;
  }
  *out = g_workspace_addr[dev];
  return TBE_OK;
}
}  // namespace

extern "C" int tbe_backward_static_workspace(const tbe_plan* plan, const float* grad_out,
                                             const int64_t* indices, int64_t N, const int64_t* offsets,
                                             int32_t B, const float* per_sample_weights,
                                             int64_t* unique_rows, int32_t* run_starts,
                                             int32_t* sorted_positions, float* row_grads,
                                             int64_t row_grads_capacity, int64_t* unique_count,
                                             int32_t* dev_status, void* stream) {
  if (!plan || B < 0 || N < 0) return TBE_ERR_INVALID_ARG;
  // a batch whose scratch does not fit the fixed array is refused up front
  if (tbe_backward_workspace_bytes(plan, B, N) > (size_t)TBE_STATIC_WORKSPACE_BYTES) return TBE_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = static_workspace(&ws);
  if (st != TBE_OK) return st;
  return tbe_backward(plan, grad_out, indices, N, offsets, B, per_sample_weights, unique_rows, run_starts,
                      sorted_positions, row_grads, row_grads_capacity, unique_count, ws,
                      (size_t)TBE_STATIC_WORKSPACE_BYTES, dev_status, stream);
}
