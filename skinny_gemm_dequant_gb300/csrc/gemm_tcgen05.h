// tcgen05 block-scaled GEMM path (M >= 17 tokens, 1x128 E4M3 activations): host interface.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ql {
namespace tc {

struct GemmArgs {
  int M, N, K;
  const uint8_t* w;   // FP8: E4M3 [N, ldw]; FP4: packed E2M1 [N, ldw] bytes
  int64_t ldw;        // bytes per weight row
  const uint8_t* ws;  // FP8: UE8M0 [ceil(N/128), lds]; FP4: UE8M0 [N, lds]
  int64_t lds;
  int fp4;
  uint8_t* aq;        // activation codes (workspace)
  uint8_t* as;        // activation scales (workspace)
  uint16_t* y;
  int64_t ldy;
  const uint16_t* bias;
  uint32_t* status;
  uint32_t wait_limit;
};

size_t act_q_bytes(int64_t M, int64_t K);
size_t act_s_bytes(int64_t M, int64_t K);
cudaError_t quantize_activations(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const GemmArgs& g,
                                 uint8_t* aq_dbg, uint8_t* as_dbg, cudaStream_t st);
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st);

}  // namespace tc
}  // namespace ql
