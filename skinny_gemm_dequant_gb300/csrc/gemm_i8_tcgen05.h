// INT8 W8A8 GEMM for M = 17..256 on tcgen05 (kind::f16 on exact f16 images of the int8 values,
// drained to int32 every 512 K): per-token activation quantisation launch + the GEMM launch.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ql {
namespace tc {

struct I8GemmArgs {
  int M, N, K;
  const uint16_t* x;  // bf16 [M, ldx]
  int64_t ldx;
  const int8_t* w;  // int8 [N, ldw]
  int64_t ldw;
  const float* w_s;  // fp32 [w_s_len], w_s_len = N or 1
  int w_s_len;
  const uint16_t* bias;  // bf16 [N] or null
  uint16_t* y;           // bf16 [M, ldy], or null (a K shard: acc_out only)
  int64_t ldy;
  int32_t* acc_out;  // optional int32 [M, N]
  int8_t* xq_dbg;    // optional int8 [M, K]
  float* xs_dbg;     // optional fp32 [M]
  uint16_t* img;     // workspace: f16 activation codes [M, kpad], kpad = K rounded up to 64
  float* xs;         // workspace: fp32 [M]
  int32_t* part;     // workspace: int32 [ks][M][N] split-K partial sums (ks = i8_splits > 1)
  unsigned* tickets; // workspace: one arrival count per output tile, zero between calls
  uint32_t* status;
  uint32_t wait_limit;
  const float* amax_in;  // optional fp32 [M]: per-token amax over the whole row (a K shard)
};

int64_t i8_kpad(int64_t K);
size_t i8_image_bytes(int64_t M, int64_t K);
// K splits of a call: more than one only when its output tiles would leave most SMs idle
int i8_splits(int64_t M, int64_t N, int64_t K);
size_t i8_part_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_i8_gemm(const I8GemmArgs& g, cudaStream_t st);

}  // namespace tc
}  // namespace ql
