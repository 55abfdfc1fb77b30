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
  // grouped (MoE) launch: one weight matrix per expert, token tiles from a device-built list
  int grouped;
  int experts;
  int64_t w_estride;       // bytes between two experts' weight matrices
  int64_t s_estride;       // bytes between two experts' weight-scale arrays
  const int4* tiles;       // (expert, first dispatch row, rows, 0)
  const int* ntiles;       // number of valid tiles (device)
  int tiles_max;           // host bound on *ntiles (grid height)
  int tt;                  // token columns per tile (16..128, a multiple of 16)
  const int32_t* pairs;    // dispatch row -> pair
  float* out;              // fp32 [pairs][ld_out]
  int64_t ld_out;
};

size_t act_q_bytes(int64_t M, int64_t K);
size_t act_s_bytes(int64_t M, int64_t K);
cudaError_t quantize_activations(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const GemmArgs& g,
                                 uint8_t* aq_dbg, uint8_t* as_dbg, cudaStream_t st);
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st);

}  // namespace tc
}  // namespace ql
