// The bf16 instances of the tcgen05 GEMM (kernel template in gemm_kernel.cuh).
#include "gemm_kernel.cuh"

namespace dit {

cudaError_t launch_gemm(int epi, int hd, const void* A, long long lda, const void* B,
                        long long ldb, GemmParams& p, cudaStream_t st) {
  return launch_gemm_t<false>(epi, hd, A, lda, B, ldb, p, st);
}

}  // namespace dit
