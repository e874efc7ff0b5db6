// The e4m3 instances of the tcgen05 GEMM (kernel template in gemm_kernel.cuh):
// 8-bit codes of both operands, fp32 scales per row of each applied in the
// epilogue.
#include "gemm_kernel.cuh"

namespace dit {

cudaError_t launch_gemm_f8(int epi, int hd, const void* A, long long lda, const void* B,
                           long long ldb, GemmParams& p, cudaStream_t st) {
  if (p.sa == nullptr || p.sb == nullptr) return cudaErrorInvalidValue;
  return launch_gemm_t<true>(epi, hd, A, lda, B, ldb, p, st);
}

}  // namespace dit
