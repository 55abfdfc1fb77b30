// INT8 W8A8 linear for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: plain C hosts without a device
// allocator of their own, plugins living inside a framework that has already reserved all
// of the GPU's memory for its own pool and forbids further cudaMalloc calls, and latency-
// critical paths that must not call cudaMalloc/cudaFree because those calls can synchronise
// the whole device.  For them this entry point takes its scratch (the quantised activations,
// the split-K partial sums and tickets) from one fixed array in the library's own device
// memory instead of from a caller-provided workspace.
//
// The array is a file-scope __device__ variable of kScratchBytes; every GPU that loads the
// library holds it until the process exits.  Its host-side name is only a stand-in for the
// device address, so the address is looked up (cudaGetSymbolAddress) on the first call made
// on each device, with that device current, and cached.  That first call therefore does a
// little set-up work and should come before any stream capture.
//
// All calls on a device share the one array and it keeps whatever the previous call left
// there: the part that must start at zero (the status word, the counters and all split-K
// tickets) is cleared on the caller's stream at the start of every call, and two calls that
// overlap on the GPU (different streams, no ordering between them) race on the array.
#include <mutex>

#include "../../include/qlinear.h"
#include "internal.h"
#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB: room for the split-K partial sums of the M > 16 GEMM
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// device address of the scratch array on the current device (set up once per device)
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ql_status qlinear_int8_w8a8_noalloc(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                               const int8_t* w, int64_t N, int64_t ldw, const float* w_scale,
                                               int64_t w_scale_len, const uint16_t* bias, uint16_t* y, int64_t ldy,
                                               int32_t* acc_out, int8_t* xq_out, float* xs_out, ql_stream_t stream,
                                               int* path_out) {
  if (path_out) *path_out = QL_PATH_NONE;
  if (M < 1 || N < 1 || K < 1) return QL_ERR_INVALID_ARG;
  const size_t need = ql_workspace_bytes(QL_OP_INT8_W8A8, M, N, K, 0, 0);
  if (need == 0 || need > kScratchBytes) return QL_ERR_WORKSPACE;  // larger than the built-in scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return QL_ERR_CUDA;
  // everything the kernels expect to find zero, whatever an earlier call (cut short by a
  // timed-out wait, say) left behind
  const size_t clear = ql::workspace_zero_bytes();
  if (cudaMemsetAsync(scratch, 0, clear, (cudaStream_t)stream) != cudaSuccess) return QL_ERR_CUDA;
  return qlinear_int8_w8a8(x, M, K, ldx, w, N, ldw, w_scale, w_scale_len, bias, y, ldy, acc_out, xq_out, xs_out,
                           scratch, kScratchBytes, stream, path_out);
}
