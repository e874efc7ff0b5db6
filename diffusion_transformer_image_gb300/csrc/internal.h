// Host-side declarations shared by the translation units of libdit.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "dit.h"

namespace dit {

// Per-device state, initialised on first use with that device current.
struct DeviceState {
  int sm_count;
  int* err;                        // device error word (a __device__ variable)
  unsigned long long timeout_ns;   // bound of every in-kernel wait
};
const DeviceState* device_state();  // nullptr if CUDA is unusable
inline DevErr dev_err(const DeviceState* ds) { return DevErr{ds->err, ds->timeout_ns}; }
void count_launch(int n = 1);

// Launches a kernel with programmatic stream serialization (see
// grid_dep_wait in common.cuh): the launch of the next kernel overlaps the
// tail of the one before it.  cluster_x > 1 adds a cluster dimension.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     int cluster_x, Args... args) {
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Encodes a row-major tensor map with 128-byte swizzle (or none): bf16
// elements (elem_bytes 2), fp32 (4) or bytes (1, the e4m3 codes).
// dims[0] is the contiguous dimension; strides_bytes has rank-1 entries.
bool make_tmap(CUtensorMap* map, uint32_t elem_bytes, const void* base, int rank,
               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
               bool swizzle128 = true);
inline bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
  return make_tmap(map, 2, base, rank, dims, strides_bytes, box);
}

// ------------------------------------------------------------------ GEMM
enum GemmEpi : int {
  EPI_BF16 = 0,       // out bf16 = acc
  EPI_F32_BIAS = 1,   // out fp32 = acc + bias
  EPI_RESIDUAL = 2,   // out fp32 += gate * acc
  EPI_SWIGLU = 3,     // out bf16 = silu(acc_gate) * acc_up
  EPI_QKV = 4,        // qk-norm + RoPE -> qk buffer; v -> transposed buffer
  EPI_GEGLU = 5,      // out bf16 = gelu_tanh_clamped(acc_gate) * acc_up
  EPI_RESIDUAL_TANH = 6,     // out fp32 += tanh(gate) * acc
  EPI_RESIDUAL_SIGMOID = 7,  // out fp32 += sigmoid(gate) * acc
  EPI_EULER = 8              // v = out + acc (out fp32, rewritten); aux += scalar * v
};

struct QkvEpi {
  __nv_bfloat16* qk;   // [nh + nkv][M][hd], q heads then k heads
  __nv_bfloat16* vt;   // [n_seqs, nkv, hd, s_pad]
  int s_len, s_pad;
  int nh, nkv;
  const float *qg, *qb, *kg, *kb;   // null when there is no qk norm
  const float *rcos, *rsin;         // pair-major [hd/2][s_len]
  int rope_half;                    // 0: pairs (2k, 2k+1); 1: pairs (k, k + hd/2)
  int rms;                          // qk-norm is RMSNorm instead of LayerNorm
  int rope_first;                   // RoPE before the qk-norm
  float eps;
};

struct GemmParams {
  int M, N, K;          // output columns N (SwiGLU: F, the h width)
  int num_m, num_n;
  void* out;
  long long ldo;
  const float* vec;     // bias (EPI_F32_BIAS) or gate (EPI_RESIDUAL), may be null
  const float* sa;      // e4m3 GEMM: scale of each A row [M]
  const float* sb;      // e4m3 GEMM: scale of each B row [N] (GLU: [2N])
  float* aux;           // EPI_EULER: the latent [M, ldo] updated in place
  float scalar;         // EPI_EULER: sigma_next - sigma
  QkvEpi qkv;
  DevErr err;
  int group_m;          // row blocks per raster group (tiles walk rows fastest inside one)
  // B is not written by the kernel launched just before this one in the
  // stream (the projections inside a block, whose weights only the caller
  // writes, before the block's first kernel): the producer may request the
  // first stages' B tiles before the grid-dependency wait.  Such a GEMM
  // starts only once every CTA of the kernel before it has passed its own
  // wait, i.e. once everything earlier has completed.
  int b_early;
};

// D = A[M,K] B[rows,K]^T with the epilogue `epi`; hd selects the QKV head
// width (64 or 128).  Returns cudaSuccess or the launch error.
cudaError_t launch_gemm(int epi, int hd, const void* A, long long lda, const void* B,
                        long long ldb, GemmParams& p, cudaStream_t st);
// The same with e4m3 codes for A and B (lda, ldb in elements = bytes) and the
// row scales p.sa, p.sb applied to the accumulator before the epilogue.
cudaError_t launch_gemm_f8(int epi, int hd, const void* A, long long lda, const void* B,
                           long long ldb, GemmParams& p, cudaStream_t st);

// ------------------------------------------------------------- attention
cudaError_t launch_attention(int hd, const __nv_bfloat16* qk, const __nv_bfloat16* vt,
                             int n_tokens, int n_seqs, int nh, int nkv, __nv_bfloat16* o,
                             cudaStream_t st);

// ------------------------------------------------------------- row ops
// mode: bit 0 affine (else AdaLN), bit 1 RMSNorm (else LayerNorm)
cudaError_t launch_ln_modulate(int mode, const float* x, long long ldx, int rows, int H,
                               const float* p0, const float* p1, float eps,
                               __nv_bfloat16* out, long long ldo, cudaStream_t st,
                               __nv_bfloat16* out_lo = nullptr);
// W8A8 coding ([ZFLOW] section VII): rows rotated by the 256-point Hadamard
// matrix along K, then e4m3 codes with one fp32 scale per row.  K (or H) a
// multiple of 256; codes [rows, ldq] bytes, scale [rows].
constexpr int ROTQ_MAX_K = 16384;
constexpr int ROTQ_LN_MAX_H = 8192;
cudaError_t launch_rotate_quant(const __nv_bfloat16* x, long long ldx, int rows, int K,
                                uint8_t* q, long long ldq, float* scale, cudaStream_t st);
// The same applied to launch_ln_modulate's output (same mode bits), which is
// never written in bf16.
cudaError_t launch_ln_rotate_quant(int mode, const float* x, long long ldx, int rows, int H,
                                   const float* p0, const float* p1, float eps, uint8_t* q,
                                   long long ldq, float* scale, cudaStream_t st);
cudaError_t launch_euler(float* x, const float* v, long long n, float dt, cudaStream_t st);
// Longest input vector of the M = 1 linears (staged whole in shared memory).
constexpr int GEMV_MAX_K = 16384;
cudaError_t launch_gemv(const __nv_bfloat16* W, const float* x, const float* b, float* y,
                        int O, int K, int silu_in, cudaStream_t st);
cudaError_t launch_sinusoid(float T, int dim, float* out, cudaStream_t st);
cudaError_t launch_rope_grid(int grid_h, int grid_w, int n_txt, const int* pos,
                             int n_pos, const int32_t* axes, float theta, int half_d,
                             float* cos_out, float* sin_out, cudaStream_t st);
cudaError_t launch_rope_vit(int grid_h, int grid_w, int n_prefix, int head_dim, float base,
                            float* cos_out, float* sin_out, cudaStream_t st);
cudaError_t launch_f32_to_bf16(const float* in, __nv_bfloat16* out, long long n,
                               cudaStream_t st);
cudaError_t launch_split_bf16(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, long long n,
                              cudaStream_t st);
cudaError_t launch_bf16_to_f32(const __nv_bfloat16* in, float* out, long long n,
                               cudaStream_t st);
cudaError_t launch_stuck_wait(DevErr e, cudaStream_t st);

}  // namespace dit
