// The W8A8 format's coding kernels ([ZFLOW] "From Python + CUDA to Pure Rust +
// Metal 4", section VII: 8-bit codes per row on both operands, a 256-point
// Hadamard rotation H256 on both sides, correct because (x H)(W H)^T = x W^T
// for orthogonal H).
//
// Each row is rotated in independent blocks of 256 along K by the Sylvester
// Hadamard matrix scaled by 1/16, then coded in e4m3 with one fp32 scale:
// amax = max |y|, scale = amax / 448, code = e4m3(y * (448 / amax)) rounded
// to nearest even and saturated.  The rotation is the fast Walsh-Hadamard
// transform with the butterfly spans in the order 1, 2, ..., 128, every
// butterfly one fp32 add or subtract, so the result does not depend on how
// the spans are spread over threads.
//
//   rotq_tma_kernel     bf16 rows (weights offline; attention output and GLU
//                       output online) -> codes + scales
//   ln_rotq_tma_kernel  the fp32 residual rows through LayerNorm/RMSNorm and
//                       the AdaLN or affine modulation, then rotated and
//                       coded: the A operand of the QKV and gate/up
//                       projections written once, in 8 bits
// Both are persistent: a ring of whole rows in shared memory filled by one
// TMA copy per row (128-byte swizzle, so that the reads below are free of
// bank conflicts), one row per pass of the CTA.  The normed rows take H / 32
// threads, each owning 32 consecutive values: spans 1..16 inside the thread
// (packed fp32 pairs from span 2), spans 32, 64, 128 between the 8 threads
// of a 256-block.  The bf16 rows take K / 64 threads of 64 values (spans
// 1..32 inside, 64 and 128 between 4 threads) when K is a multiple of 2048,
// else K / 32 of 32: these kernels are bound by their instruction count and
// per-row latency rather than by HBM, and an exchange span costs three
// times an in-thread one per value.
// One barrier per row for the bf16 rows (three for the normed rows: mean,
// variance, maximum).  Rows whose K is not a multiple of 1024 (or too long)
// take the warp-per-block kernels rotq_kernel / ln_rotq_kernel instead.
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
  grid_dep_wait();
  grid_dep_launch();
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
  grid_dep_wait();
  grid_dep_launch();
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

// ------------------------------------------------------------ TMA-ring kernels
constexpr int RQT_MAX_THREADS = 512;     // K <= 16384
constexpr int RQT_LN_MAX_THREADS = 256;  // H <= 8192
// Rows in flight per CTA.  A CTA codes its rows one after another behind
// block barriers, so the kernels are bound by that chain's latency unless
// many CTAs share an SM: a two-row ring keeps the shared memory per CTA
// small (for 4096-wide rows 9 bf16 or 4 fp32 CTAs per SM, then limited by
// registers), and 2 x (CTAs per SM) rows are still in flight per SM.
constexpr int RQT_STAGES = 2;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

// The exact scaling by 1/16 that ends the rotation, on packed pairs.  (It
// stays a multiplication of every value: moving it to the row scale gives
// the same bits only while the rotated values are normal floats.)
template <int N>
__device__ __forceinline__ void scale_sixteenth(float (&v)[N]) {
  const float2 sixteenth = make_float2(0.0625f, 0.0625f);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float2 r = __fmul2_rn(make_float2(v[i], v[i + 1]), sixteenth);
    v[i] = r.x;
    v[i + 1] = r.y;
  }
}

// x H over this thread's 32 values (elements 32 j + e of a 256-block, j =
// lane % 8), spans 1, 2, ..., 128 in order; then the exact scaling by 1/16.
__device__ __forceinline__ void fwht256_seg32(float (&v)[32], int lane) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {  // span 1
    const float a = v[i], b = v[i + 1];
    v[i] = a + b;
    v[i + 1] = a - b;
  }
  const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {  // spans 2, 4, 8, 16 on pairs (2j, 2j+1)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (!(j & h)) {
        const float2 a = make_float2(v[2 * j], v[2 * j + 1]);
        const float2 b = make_float2(v[2 * (j + h)], v[2 * (j + h) + 1]);
        const float2 s = __fadd2_rn(a, b);
        const float2 d = __ffma2_rn(b, neg1, a);  // a - b, one rounding
        v[2 * j] = s.x;
        v[2 * j + 1] = s.y;
        v[2 * (j + h)] = d.x;
        v[2 * (j + h) + 1] = d.y;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {  // spans 32, 64, 128 between lanes
    const float sg = (lane & m) ? -1.0f : 1.0f;  // upper index: partner - mine
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[i], m),
                                   __shfl_xor_sync(0xffffffffu, v[i + 1], m));
      const float2 r = __ffma2_rn(sg2, make_float2(v[i], v[i + 1]), o);
      v[i] = r.x;
      v[i + 1] = r.y;
    }
  }
  scale_sixteenth(v);
}

// The same for 64 values per thread (elements 64 j + e, j = lane % 4):
// spans 1..32 inside the thread, 64 and 128 between the 4 lanes of a block.
// Fewer instructions per element than 32 values per thread (one exchange
// span less), which is what bounds these kernels.
__device__ __forceinline__ void fwht256_seg64(float (&v)[64], int lane) {
#pragma unroll
  for (int i = 0; i < 64; i += 2) {  // span 1
    const float a = v[i], b = v[i + 1];
    v[i] = a + b;
    v[i + 1] = a - b;
  }
  const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {  // spans 2, 4, 8, 16, 32 on pairs (2j, 2j+1)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (!(j & h)) {
        const float2 a = make_float2(v[2 * j], v[2 * j + 1]);
        const float2 b = make_float2(v[2 * (j + h)], v[2 * (j + h) + 1]);
        const float2 s = __fadd2_rn(a, b);
        const float2 d = __ffma2_rn(b, neg1, a);
        v[2 * j] = s.x;
        v[2 * j + 1] = s.y;
        v[2 * (j + h)] = d.x;
        v[2 * (j + h) + 1] = d.y;
      }
    }
  }
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {  // spans 64, 128 between lanes
    const float sg = (lane & m) ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, v[i], m),
                                   __shfl_xor_sync(0xffffffffu, v[i + 1], m));
      const float2 r = __ffma2_rn(sg2, make_float2(v[i], v[i + 1]), o);
      v[i] = r.x;
      v[i + 1] = r.y;
    }
  }
  scale_sixteenth(v);
}

// max |v[i]| over an array, two values per three-input maximum
template <int N>
__device__ __forceinline__ float abs_max(const float (&v)[N]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < N; i += 2) m = fmax3(m, fabsf(v[i]), fabsf(v[i + 1]));
  return m;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Codes this thread's N rotated values with the row's maximum and stores
// the N bytes at dst; thread 0 stores the scale.
template <int N>
__device__ __forceinline__ void code_seg(const float (&v)[N], float amax, uint8_t* dst,
                                         float* scale_out) {
  const float inv = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 0.0f;
  if (threadIdx.x == 0) *scale_out = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 0.0f;
  const float2 inv2 = make_float2(inv, inv);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < N / 16; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 16 * c + 4 * q;
      const float2 a = __fmul2_rn(make_float2(v[i], v[i + 1]), inv2);
      const float2 b = __fmul2_rn(make_float2(v[i + 2], v[i + 3]), inv2);
      w[q] = pack_e4m3x4(a.x, a.y, b.x, b.y);
    }
    d[c] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Issues the TMA copy of row `row` into ring stage `s` (one elected thread).
__device__ __forceinline__ void rqt_issue(uint8_t* smem, int row_bytes, uint64_t* full, int s,
                                          const CUtensorMap* tm, int row) {
  mbar_arrive_expect_tx(&full[s], (uint32_t)row_bytes);
  tma_load_3d(smem + (size_t)s * row_bytes, tm, &full[s], 0, 0, row);
}

// After a wait that ran out: every copy still in flight must land before the
// CTA may exit.  Rows n in [first, issued) of this CTA went to stage n % S.
__device__ __forceinline__ void rqt_drain(uint64_t* full, int first, int issued, const DevErr& e) {
  for (int n = first; n < issued; ++n)
    mbar_wait(&full[n % RQT_STAGES], (uint32_t)((n / RQT_STAGES) & 1), e);
}

// bf16 rows [rows, K] (3-D map: 64 x K/64 x rows, box one row) -> codes,
// K / VPT threads of VPT consecutive values each (VPT = 64 when K is a
// multiple of 2048, else 32).
template <int VPT>
__global__ void __launch_bounds__(16384 / VPT) rotq_tma_kernel(
    const __grid_constant__ CUtensorMap tm, int rows, int K, uint8_t* __restrict__ q,
    long long ldq, float* __restrict__ scale, DevErr err) {
  static_assert(VPT == 32 || VPT == 64, "32 or 64 values per thread");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int row_bytes = K * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)RQT_STAGES * row_bytes);
  __shared__ float red[2][RQT_MAX_THREADS / 32];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, nwarps = blockDim.x >> 5;
  const int G = gridDim.x;
  int issued = 0;  // rows of this CTA whose copy has been issued (thread 0)
  grid_dep_wait();
  grid_dep_launch();
  if (t == 0) {
    for (int s = 0; s < RQT_STAGES; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm);
    for (int s = 0; s < RQT_STAGES && blockIdx.x + s * G < rows; ++s, ++issued)
      rqt_issue(smem, row_bytes, full, s, &tm, blockIdx.x + s * G);
  }
  __syncthreads();
  // this thread's 2 VPT bytes: 16-byte chunks c0 .. c0 + VPT / 8 - 1 of the
  // 128-byte line L (chunk c of line L sits at c ^ (L % 8): 128-byte swizzle)
  constexpr int TPL = 64 / VPT;  // threads per line
  const int L = t / TPL, c0 = (t % TPL) * (VPT / 8);
  int it = 0;
  for (int row = blockIdx.x; row < rows; row += G, ++it) {
    const int s = it % RQT_STAGES;
    const bool ok = mbar_wait(&full[s], (uint32_t)((it / RQT_STAGES) & 1), err);
    float v[VPT];
    const uint8_t* line = smem + (size_t)s * row_bytes + (size_t)L * 128;
#pragma unroll
    for (int k = 0; k < VPT / 8; ++k) {
      const uint4 u = *reinterpret_cast<const uint4*>(line + (((c0 + k) ^ (L & 7)) << 4));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * k + 2 * i] = __uint_as_float(w[i] << 16);
        v[8 * k + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
    if constexpr (VPT == 64)
      fwht256_seg64(v, lane);
    else
      fwht256_seg32(v, lane);
    float m = warp_max(abs_max(v));
    if (lane == 0) red[it & 1][warp] = m;
    // every thread has read stage s and published its maximum
    if (!__syncthreads_and(ok)) {
      if (t == 0) rqt_drain(full, it, issued, err);
      break;
    }
    if (t == 0 && row + RQT_STAGES * G < rows) {
      rqt_issue(smem, row_bytes, full, s, &tm, row + RQT_STAGES * G);
      ++issued;
    }
    float amax = red[it & 1][0];
    for (int w2 = 1; w2 < nwarps; ++w2) amax = fmaxf(amax, red[it & 1][w2]);
    code_seg<VPT>(v, amax, q + (size_t)row * ldq + (size_t)t * VPT, scale + row);
  }
}

// fp32 rows [rows, H] (3-D map: 32 x H/32 x rows) through the norm and the
// modulation, rotated and coded.  MODE bit 0: affine n g + b (else AdaLN
// n (1 + scale) + shift); RMS: RMSNorm.
template <int MODE, bool RMS>
__global__ void __launch_bounds__(RQT_LN_MAX_THREADS) ln_rotq_tma_kernel(
    const __grid_constant__ CUtensorMap tm, int rows, int H, const float* __restrict__ p0,
    const float* __restrict__ p1, float eps, uint8_t* __restrict__ q, long long ldq,
    float* __restrict__ scale, DevErr err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int row_bytes = H * 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)RQT_STAGES * row_bytes);
  __shared__ float red_s[RQT_MAX_THREADS / 32], red_v[RQT_MAX_THREADS / 32],
      red_m[RQT_MAX_THREADS / 32];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, nwarps = blockDim.x >> 5;
  const int G = gridDim.x;
  int issued = 0;
  grid_dep_wait();
  grid_dep_launch();
  if (t == 0) {
    for (int s = 0; s < RQT_STAGES; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm);
    for (int s = 0; s < RQT_STAGES && blockIdx.x + s * G < rows; ++s, ++issued)
      rqt_issue(smem, row_bytes, full, s, &tm, blockIdx.x + s * G);
  }
  // this thread's modulation parameters (32 consecutive columns), kept in
  // registers for every row (read per row they would come from L2: the L1
  // left beside the CTAs' rings is smaller than the two vectors)
  float pa[32], pb[32];
  {
    const float4* a4 = reinterpret_cast<const float4*>(p0 + (size_t)t * 32);
    const float4* b4 = reinterpret_cast<const float4*>(p1 + (size_t)t * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 a = __ldg(a4 + i), b = __ldg(b4 + i);
      pa[4 * i] = a.x; pa[4 * i + 1] = a.y; pa[4 * i + 2] = a.z; pa[4 * i + 3] = a.w;
      pb[4 * i] = b.x; pb[4 * i + 1] = b.y; pb[4 * i + 2] = b.z; pb[4 * i + 3] = b.w;
    }
  }
  __syncthreads();
  int it = 0;
  for (int row = blockIdx.x; row < rows; row += G, ++it) {
    const int s = it % RQT_STAGES;
    const bool ok = mbar_wait(&full[s], (uint32_t)((it / RQT_STAGES) & 1), err);
    float v[32];
    const uint8_t* line = smem + (size_t)s * row_bytes + (size_t)t * 128;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const float4 f = *reinterpret_cast<const float4*>(line + ((p ^ (t & 7)) << 4));
      v[4 * p] = f.x; v[4 * p + 1] = f.y; v[4 * p + 2] = f.z; v[4 * p + 3] = f.w;
    }
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) sum += v[i];
    sum = warp_sum(sum);
    if (lane == 0) red_s[warp] = sum;
    if (!__syncthreads_and(ok)) {
      if (t == 0) rqt_drain(full, it, issued, err);
      break;
    }
    // stage s is free again
    if (t == 0 && row + RQT_STAGES * G < rows) {
      rqt_issue(smem, row_bytes, full, s, &tm, row + RQT_STAGES * G);
      ++issued;
    }
    float mean = 0.f;
    if (!RMS) {
      for (int w2 = 0; w2 < nwarps; ++w2) mean += red_s[w2];
      mean /= (float)H;
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] -= mean;
      ss = fmaf(v[i], v[i], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red_v[warp] = ss;
    __syncthreads();
    float var = 0.f;
    for (int w2 = 0; w2 < nwarps; ++w2) var += red_v[w2];
    const float rstd = 1.0f / sqrtf(var / (float)H + eps);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float n = v[i] * rstd;
      v[i] = (MODE & 1) ? fmaf(n, pa[i], pb[i]) : fmaf(n, 1.0f + pb[i], pa[i]);
    }
    fwht256_seg32(v, lane);
    float m = warp_max(abs_max(v));
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    float amax = red_m[0];
    for (int w2 = 1; w2 < nwarps; ++w2) amax = fmaxf(amax, red_m[w2]);
    code_seg<32>(v, amax, q + (size_t)row * ldq + (size_t)t * 32, scale + row);
  }
}

size_t rqt_smem_bytes(int row_bytes) {
  return (size_t)RQT_STAGES * row_bytes + 1024 + RQT_STAGES * sizeof(uint64_t) + 64;
}

// Persistent grid: as many CTAs as fit on an SM (queried once per device,
// kernel variant and row length), times the SMs, at most one per row.
template <typename Kern>
cudaError_t rqt_grid(Kern kern, int variant, int threads, int row_bytes, int rows, int* grid) {
  constexpr int MAXDEV = 64, VARIANTS = 6, LENGTHS = 33;
  static int occ[MAXDEV][VARIANTS][LENGTHS];
  static bool attr[MAXDEV][VARIANTS];
  const DeviceState* ds = device_state();
  int dev = 0;
  if (!ds || cudaGetDevice(&dev) != cudaSuccess || dev >= MAXDEV) return cudaErrorInitializationError;
  const int li = row_bytes / 2048;  // row_bytes is a multiple of 2048, at most 65536
  if (variant >= VARIANTS || li >= LENGTHS) return cudaErrorInvalidValue;
  const size_t smem = rqt_smem_bytes(row_bytes);
  if (!attr[dev][variant]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rqt_smem_bytes(32768));
    if (e != cudaSuccess) return e;
    attr[dev][variant] = true;
  }
  if (occ[dev][variant][li] == 0) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    occ[dev][variant][li] = per_sm;
  }
  const long long cap = (long long)occ[dev][variant][li] * ds->sm_count;
  *grid = (int)(rows < cap ? rows : cap);
  return cudaSuccess;
}

template <int MODE, bool RMS>
cudaError_t ln_rotq_tma_launch(const CUtensorMap& tm, int rows, int H, const float* p0,
                               const float* p1, float eps, uint8_t* q, long long ldq,
                               float* scale, cudaStream_t st) {
  const int threads = H / 32, row_bytes = H * 4;
  int grid = 0;
  cudaError_t e = rqt_grid(ln_rotq_tma_kernel<MODE, RMS>, 1 + MODE + (RMS ? 2 : 0), threads,
                           row_bytes, rows, &grid);
  if (e != cudaSuccess) return e;
  return launch_k(ln_rotq_tma_kernel<MODE, RMS>, dim3(grid), dim3(threads),
                  rqt_smem_bytes(row_bytes), st, 1, tm, rows, H, p0, p1, eps, q, ldq, scale,
                  dev_err(device_state()));
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int MAXC>
cudaError_t rotq_launch(const __nv_bfloat16* x, long long ldx, int rows, int K, uint8_t* q,
                        long long ldq, float* scale, cudaStream_t st) {
  return launch_k(rotq_kernel<MAXC>, dim3(rows), dim3(RQ_THREADS), 0, st, 1, x, ldx, rows, K, q,
                  ldq, scale);
}

template <int MODE, bool RMS, int MAXC>
cudaError_t ln_rotq_launch(const float* x, long long ldx, int rows, int H, const float* p0,
                           const float* p1, float eps, uint8_t* q, long long ldq, float* scale,
                           cudaStream_t st) {
  return launch_k(ln_rotq_kernel<MODE, RMS, MAXC>, dim3(rows), dim3(RQ_THREADS), 0, st, 1, x,
                  ldx, rows, H, p0, p1, eps, q, ldq, scale);
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
  if (K % 1024 == 0) {  // the TMA-ring kernel: K / 64 or K / 32 threads, one 3-D copy per row
    CUtensorMap tm;
    const uint64_t dims[3] = {64, (uint64_t)K / 64, (uint64_t)rows};
    const uint64_t strides[2] = {128, (uint64_t)ldx * 2};
    const uint32_t box[3] = {64, (uint32_t)K / 64, 1};
    if (!make_tmap(&tm, 2, x, 3, dims, strides, box)) return cudaErrorInvalidValue;
    int grid = 0;
    const DevErr err = dev_err(device_state());
    if (K % 2048 == 0) {
      cudaError_t e = rqt_grid(rotq_tma_kernel<64>, 5, K / 64, K * 2, rows, &grid);
      if (e != cudaSuccess) return e;
      return launch_k(rotq_tma_kernel<64>, dim3(grid), dim3(K / 64), rqt_smem_bytes(K * 2), st, 1,
                      tm, rows, K, q, ldq, scale, err);
    }
    cudaError_t e = rqt_grid(rotq_tma_kernel<32>, 0, K / 32, K * 2, rows, &grid);
    if (e != cudaSuccess) return e;
    return launch_k(rotq_tma_kernel<32>, dim3(grid), dim3(K / 32), rqt_smem_bytes(K * 2), st, 1,
                    tm, rows, K, q, ldq, scale, err);
  }
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
  if (H % 1024 == 0) {  // the TMA-ring kernel: H / 32 threads, one 3-D copy per row
    CUtensorMap tm;
    const uint64_t dims[3] = {32, (uint64_t)H / 32, (uint64_t)rows};
    const uint64_t strides[2] = {128, (uint64_t)ldx * 4};
    const uint32_t box[3] = {32, (uint32_t)H / 32, 1};
    if (!make_tmap(&tm, 4, x, 3, dims, strides, box)) return cudaErrorInvalidValue;
    switch (mode) {
      case 0: return ln_rotq_tma_launch<0, false>(tm, rows, H, p0, p1, eps, q, ldq, scale, st);
      case 1: return ln_rotq_tma_launch<1, false>(tm, rows, H, p0, p1, eps, q, ldq, scale, st);
      case 2: return ln_rotq_tma_launch<0, true>(tm, rows, H, p0, p1, eps, q, ldq, scale, st);
      default: return ln_rotq_tma_launch<1, true>(tm, rows, H, p0, p1, eps, q, ldq, scale, st);
    }
  }
  switch (mode) {
    case 0: return ln_rotq_dispatch<0, false>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
    case 1: return ln_rotq_dispatch<1, false>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
    case 2: return ln_rotq_dispatch<0, true>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
    default: return ln_rotq_dispatch<1, true>(x, ldx, rows, H, p0, p1, eps, q, ldq, scale, st);
  }
}

}  // namespace dit
