// The W8A8 format's coding kernels ([ZFLOW] "From Python + CUDA to Pure Rust +
// Metal 4", section VII: 8-bit codes per row on both operands, a 256-point
// Hadamard rotation H256 on both sides, correct because (x H)(W H)^T = x W^T
// for orthogonal H).
//
// Each row is rotated in independent blocks of 256 along K by the Sylvester
// Hadamard matrix scaled by 1/16, then coded in e4m3 with one fp32 scale:
// amax = max |y|, scale = amax / 448, code = e4m3(y * (448 / amax)) rounded
// to nearest even and saturated.  The rotation is the fast Walsh-Hadamard
// transform: butterfly spans 1, 2 and 4 inside a thread's 8 consecutive
// values, spans 8 ... 128 between the 32 lanes of a warp, so one warp owns one
// 256-wide block and no shared memory is touched until the row maximum.
//
//   rotq_kernel     bf16 rows (weights offline; attention output and GLU
//                   output online) -> codes + scales
//   ln_rotq_kernel  the fp32 residual rows through LayerNorm/RMSNorm and the
//                   AdaLN or affine modulation, then rotated and coded: the
//                   A operand of the QKV and gate/up projections written
//                   once, in 8 bits
//
// One 256-thread block per row; the row stays in registers (K <= 256 * 8 *
// MAXC).  Loads and stores are 16- and 8-byte vectors, coalesced per warp.
#include "internal.h"

namespace dit {
namespace {

constexpr int RQ_THREADS = 256;
constexpr int RQ_WARPS = RQ_THREADS / 32;

// x H for one 256-wide block held 8 values per lane (value i of lane l is
// element 8 l + i), H the 1/16-scaled Sylvester Hadamard matrix.
__device__ __forceinline__ void fwht256_warp(float (&v)[8], int lane) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (!(i & h)) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = upper ? o - v[i] : v[i] + o;  // lower index: u + w, upper: u - w
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] *= 0.0625f;
}

__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();  // red[] may still be read by a previous reduction
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < RQ_WARPS; ++w) m = fmaxf(m, red[w]);
  return m;
}

__device__ __forceinline__ float block_sum_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return ((red[0] + red[1]) + (red[2] + red[3])) + ((red[4] + red[5]) + (red[6] + red[7]));
}

// Codes the rotated row held in v (chunk c = warp + 8 j for slot j) and
// writes codes and the row scale.
template <int MAXC>
__device__ __forceinline__ void code_row(float (&v)[MAXC][8], int nchunks, int row,
                                         uint8_t* __restrict__ q, long long ldq,
                                         float* __restrict__ scale, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    if (warp + RQ_WARPS * j < nchunks) {
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[j][i]));
    }
  }
  const float amax = block_max_256(m, red);
  const float inv = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 0.0f;
  if (threadIdx.x == 0) scale[row] = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 0.0f;
  uint8_t* qr = q + (size_t)row * ldq;
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int c = warp + RQ_WARPS * j;
    if (c < nchunks) {
      uint2 u;
      u.x = pack_e4m3x4(__fmul_rn(v[j][0], inv), __fmul_rn(v[j][1], inv),
                        __fmul_rn(v[j][2], inv), __fmul_rn(v[j][3], inv));
      u.y = pack_e4m3x4(__fmul_rn(v[j][4], inv), __fmul_rn(v[j][5], inv),
                        __fmul_rn(v[j][6], inv), __fmul_rn(v[j][7], inv));
      *reinterpret_cast<uint2*>(qr + (size_t)c * 256 + lane * 8) = u;
    }
  }
}

template <int MAXC>
__global__ void __launch_bounds__(RQ_THREADS) rotq_kernel(const __nv_bfloat16* __restrict__ x,
                                                          long long ldx, int rows, int K,
                                                          uint8_t* __restrict__ q, long long ldq,
                                                          float* __restrict__ scale) {
  __shared__ float red[RQ_WARPS];
  const int row = blockIdx.x;
  if (row >= rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = K >> 8;
  const __nv_bfloat16* xr = x + (size_t)row * ldx;
  float v[MAXC][8];
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int c = warp + RQ_WARPS * j;
    if (c < nchunks) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)c * 256 + lane * 8));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[j][2 * i] = f.x;
        v[j][2 * i + 1] = f.y;
      }
      fwht256_warp(v[j], lane);
    }
  }
  code_row<MAXC>(v, nchunks, row, q, ldq, scale, red);
}

// MODE bit 0: affine n g + b (else AdaLN n (1 + scale) + shift); RMS: RMSNorm.
template <int MODE, bool RMS, int MAXC>
__global__ void __launch_bounds__(RQ_THREADS) ln_rotq_kernel(
    const float* __restrict__ x, long long ldx, int rows, int H, const float* __restrict__ p0,
    const float* __restrict__ p1, float eps, uint8_t* __restrict__ q, long long ldq,
    float* __restrict__ scale) {
  __shared__ float red[RQ_WARPS];
  const int row = blockIdx.x;
  if (row >= rows) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = H >> 8;
  const float* xr = x + (size_t)row * ldx;
  float v[MAXC][8];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int c = warp + RQ_WARPS * j;
    if (c < nchunks) {
      const float4* src = reinterpret_cast<const float4*>(xr + (size_t)c * 256 + lane * 8);
      const float4 a = __ldg(src), b = __ldg(src + 1);
      v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
      v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[j][i];
    }
  }
  const float mean = RMS ? 0.0f : block_sum_256(s, red) / (float)H;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    if (warp + RQ_WARPS * j < nchunks) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[j][i] -= mean;
        ss = fmaf(v[j][i], v[j][i], ss);
      }
    }
  }
  const float rstd = 1.0f / sqrtf(block_sum_256(ss, red) / (float)H + eps);
#pragma unroll
  for (int j = 0; j < MAXC; ++j) {
    const int c = warp + RQ_WARPS * j;
    if (c < nchunks) {
      const size_t off = (size_t)c * 256 + lane * 8;
      const float4* a4 = reinterpret_cast<const float4*>(p0 + off);
      const float4* b4 = reinterpret_cast<const float4*>(p1 + off);
      const float4 a0 = __ldg(a4), a1 = __ldg(a4 + 1), b0 = __ldg(b4), b1 = __ldg(b4 + 1);
      const float pa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float pb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float n = v[j][i] * rstd;
        v[j][i] = (MODE & 1) ? fmaf(n, pa[i], pb[i]) : fmaf(n, 1.0f + pb[i], pa[i]);
      }
      fwht256_warp(v[j], lane);
    }
  }
  code_row<MAXC>(v, nchunks, row, q, ldq, scale, red);
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int MAXC>
cudaError_t rotq_launch(const __nv_bfloat16* x, long long ldx, int rows, int K, uint8_t* q,
                        long long ldq, float* scale, cudaStream_t st) {
  rotq_kernel<MAXC><<<rows, RQ_THREADS, 0, st>>>(x, ldx, rows, K, q, ldq, scale);
  count_launch();
  return cudaGetLastError();
}

template <int MODE, bool RMS, int MAXC>
cudaError_t ln_rotq_launch(const float* x, long long ldx, int rows, int H, const float* p0,
                           const float* p1, float eps, uint8_t* q, long long ldq, float* scale,
                           cudaStream_t st) {
  ln_rotq_kernel<MODE, RMS, MAXC>
      <<<rows, RQ_THREADS, 0, st>>>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale);
  count_launch();
  return cudaGetLastError();
}

template <int MODE, bool RMS>
cudaError_t ln_rotq_dispatch(const float* x, long long ldx, int rows, int H, const float* p0,
                             const float* p1, float eps, uint8_t* q, long long ldq, float* scale,
                             cudaStream_t st) {
  const int per_warp = (H / 256 + RQ_WARPS - 1) / RQ_WARPS;
  if (per_warp <= 1) return ln_rotq_launch<MODE, RMS, 1>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
  if (per_warp <= 2) return ln_rotq_launch<MODE, RMS, 2>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
  return ln_rotq_launch<MODE, RMS, 4>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
}

}  // namespace

cudaError_t launch_rotate_quant(const __nv_bfloat16* x, long long ldx, int rows, int K,
                                uint8_t* q, long long ldq, float* scale, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (rows < 0 || K <= 0 || K % 256 != 0 || K > ROTQ_MAX_K || ldx < K || ldq < K ||
      ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return cudaErrorInvalidValue;
  const int per_warp = (K / 256 + RQ_WARPS - 1) / RQ_WARPS;
  if (per_warp <= 1) return rotq_launch<1>(x, ldx, rows, K, q, ldq, scale, st);
  if (per_warp <= 2) return rotq_launch<2>(x, ldx, rows, K, q, ldq, scale, st);
  if (per_warp <= 4) return rotq_launch<4>(x, ldx, rows, K, q, ldq, scale, st);
  return rotq_launch<8>(x, ldx, rows, K, q, ldq, scale, st);
}

cudaError_t launch_ln_rotate_quant(int mode, const float* x, long long ldx, int rows, int H,
                                   const float* p0, const float* p1, float eps, uint8_t* q,
                                   long long ldq, float* scale, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (rows < 0 || H <= 0 || H % 256 != 0 || H > ROTQ_LN_MAX_H || ldx < H || ldq < H ||
      ldx % 4 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(p0, 16) ||
      !aligned(p1, 16) || !aligned(q, 16) || !aligned(scale, 4) || mode < 0 || mode > 3)
    return cudaErrorInvalidValue;
  switch (mode) {
    case 0: return ln_rotq_dispatch<0, false>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
    case 1: return ln_rotq_dispatch<1, false>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
    case 2: return ln_rotq_dispatch<0, true>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
    default: return ln_rotq_dispatch<1, true>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
  }
}

}  // namespace dit
