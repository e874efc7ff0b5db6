// Bandwidth-bound kernels of the path: the AdaLN LayerNorm + modulation, the
// flow-matching Euler update, the M = 1 linears of the timestep MLP and
// modulation heads, the timestep sinusoid, RoPE tables and dtype casts.
// All loads and stores are 16-byte vectors, one warp per row where a row
// reduction is needed.
#include <math_constants.h>

#include "internal.h"

namespace dit {
namespace {

// ----------------------------------------------------- LayerNorm + modulate
// LN over the row (biased variance) or RMSNorm, then AdaLN `n (1 + scale) + shift`
// ([ERNIE] "Porting ERNIE-Image-Turbo to Zig and Metal", section IV and
// section V, Bug 4; [ZFLOW] section VI `plus_one`: the 1 is added on the
// device) or the affine `n g + b` of the pre-norm ViT ([MAKEPAD]).  One
// 256-thread block per row, the row held in registers (H <= 256 * 4 * MAXV),
// mean and variance by warp shuffles plus one shared-memory exchange.  A
// 256-thread block keeps a thread's share of a 4096-wide row at four 16-byte
// vectors, so more rows are in flight per SM and the last wave of rows is a
// small part of the launch.
constexpr int LN_THREADS = 256;
constexpr int LN_WARPS = LN_THREADS / 32;
constexpr int LN_MAXV = 8;  // float4 per thread: H <= 8192 (4 for H <= 4096)

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();  // red[] may still be read by a previous call
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < LN_WARPS; ++i) t += red[i];
  return t;
}

// With `out_lo` the result is also kept to about 16 significant bits as the
// pair hi = bf16(r), lo = bf16(r - hi): two bf16 GEMMs over hi and lo then
// reproduce an fp32-input linear (used by the fp32 head and tail projections).
template <int MODE, bool RMS, int MAXV>
__global__ void __launch_bounds__(LN_THREADS) ln_modulate_kernel(
    const float* __restrict__ x, long long ldx, int rows, int H, const float* __restrict__ p0,
    const float* __restrict__ p1, float eps, __nv_bfloat16* __restrict__ out, long long ldo,
    __nv_bfloat16* __restrict__ out_lo) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float red[LN_WARPS];
  const int row = blockIdx.x;
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * ldx);
  const int n4 = H >> 2;
  float4 v[MAXV];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + LN_THREADS * i;
    if (idx < n4) {
      v[i] = __ldg(xr + idx);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
  }
  // RMSNorm keeps the mean (it divides by the root mean square instead)
  const float mean = RMS ? 0.0f : block_sum(s, red) / (float)H;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + LN_THREADS * i;
    if (idx < n4) {
      v[i].x -= mean; v[i].y -= mean; v[i].z -= mean; v[i].w -= mean;
      ss += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
    }
  }
  const float rstd = 1.0f / sqrtf(block_sum(ss, red) / (float)H + eps);
  uint2* orow = reinterpret_cast<uint2*>(out + (size_t)row * ldo);
  const float4* a4 = reinterpret_cast<const float4*>(p0);
  const float4* b4 = reinterpret_cast<const float4*>(p1);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int idx = threadIdx.x + LN_THREADS * i;
    if (idx < n4) {
      const float4 a = __ldg(a4 + idx), b = __ldg(b4 + idx);
      float4 n = v[i];
      n.x *= rstd; n.y *= rstd; n.z *= rstd; n.w *= rstd;
      float4 r;
      if (MODE == 0) {  // AdaLN: a = shift, b = scale
        r.x = fmaf(n.x, 1.0f + b.x, a.x);
        r.y = fmaf(n.y, 1.0f + b.y, a.y);
        r.z = fmaf(n.z, 1.0f + b.z, a.z);
        r.w = fmaf(n.w, 1.0f + b.w, a.w);
      } else {          // affine: a = gain, b = bias
        r.x = fmaf(n.x, a.x, b.x);
        r.y = fmaf(n.y, a.y, b.y);
        r.z = fmaf(n.z, a.z, b.z);
        r.w = fmaf(n.w, a.w, b.w);
      }
      uint2 u;
      u.x = pack_bf16x2(r.x, r.y);
      u.y = pack_bf16x2(r.z, r.w);
      orow[idx] = u;
      if (out_lo) {
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
        const float2 h0 = __bfloat1622float2(hv[0]), h1 = __bfloat1622float2(hv[1]);
        uint2 l;
        l.x = pack_bf16x2(r.x - h0.x, r.y - h0.y);
        l.y = pack_bf16x2(r.z - h1.x, r.w - h1.y);
        reinterpret_cast<uint2*>(out_lo + (size_t)row * ldo)[idx] = l;
      }
    }
  }
}

// One warp per row for narrow rows, H = 128 NV (H <= 1024): the row in 32
// lanes x NV float4, sums by shuffles only (no block barrier), the
// modulation vectors read as they are used.  Rows are independent warps, so
// an SM keeps dozens of rows in flight and none waits on another's
// reduction.  (A 4096-wide row would take 128 registers per lane and fewer
// rows per SM: the block kernel above is faster there.)
constexpr int LNW_WARPS = 4;

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int MODE, bool RMS, int NV>
__global__ void __launch_bounds__(LNW_WARPS * 32) ln_modulate_warp_kernel(
    const float* __restrict__ x, long long ldx, int rows, const float* __restrict__ p0,
    const float* __restrict__ p1, float eps, __nv_bfloat16* __restrict__ out, long long ldo,
    __nv_bfloat16* __restrict__ out_lo) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int H = 128 * NV;
  const int row = blockIdx.x * LNW_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * ldx);
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = __ldg(xr + lane + 32 * i);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  // RMSNorm keeps the mean (it divides by the root mean square instead)
  const float mean = RMS ? 0.0f : warp_allsum(s) * (1.0f / H);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    v[i].x -= mean; v[i].y -= mean; v[i].z -= mean; v[i].w -= mean;
    ss += (v[i].x * v[i].x + v[i].y * v[i].y) + (v[i].z * v[i].z + v[i].w * v[i].w);
  }
  const float rstd = 1.0f / sqrtf(warp_allsum(ss) * (1.0f / H) + eps);
  uint2* orow = reinterpret_cast<uint2*>(out + (size_t)row * ldo);
  const float4* a4 = reinterpret_cast<const float4*>(p0);
  const float4* b4 = reinterpret_cast<const float4*>(p1);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = lane + 32 * i;
    const float4 a = __ldg(a4 + idx), b = __ldg(b4 + idx);
    float4 n = v[i];
    n.x *= rstd; n.y *= rstd; n.z *= rstd; n.w *= rstd;
    float4 r;
    if (MODE == 0) {  // AdaLN: a = shift, b = scale
      r.x = fmaf(n.x, 1.0f + b.x, a.x);
      r.y = fmaf(n.y, 1.0f + b.y, a.y);
      r.z = fmaf(n.z, 1.0f + b.z, a.z);
      r.w = fmaf(n.w, 1.0f + b.w, a.w);
    } else {          // affine: a = gain, b = bias
      r.x = fmaf(n.x, a.x, b.x);
      r.y = fmaf(n.y, a.y, b.y);
      r.z = fmaf(n.z, a.z, b.z);
      r.w = fmaf(n.w, a.w, b.w);
    }
    uint2 u;
    u.x = pack_bf16x2(r.x, r.y);
    u.y = pack_bf16x2(r.z, r.w);
    orow[idx] = u;
    if (out_lo) {
      const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
      const float2 h0 = __bfloat1622float2(hv[0]), h1 = __bfloat1622float2(hv[1]);
      uint2 l;
      l.x = pack_bf16x2(r.x - h0.x, r.y - h0.y);
      l.y = pack_bf16x2(r.z - h1.x, r.w - h1.y);
      reinterpret_cast<uint2*>(out_lo + (size_t)row * ldo)[idx] = l;
    }
  }
}

// ------------------------------------------------------------------- Euler
// x <- x + (sigma_next - sigma) v, the product rounded before the add
// ([ZFLOW] section IV, Euler sign +1).
__global__ void euler_kernel(float* __restrict__ x, const float* __restrict__ v, long long n,
                             float dt) {
  grid_dep_wait();
  grid_dep_launch();
  const long long n4 = n >> 2;
  const long long stride = (long long)gridDim.x * blockDim.x;
  float4* x4 = reinterpret_cast<float4*>(x);
  const float4* v4 = reinterpret_cast<const float4*>(v);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 a = __ldcs(x4 + i);
    const float4 b = __ldcs(v4 + i);
    a.x = __fadd_rn(a.x, __fmul_rn(dt, b.x));
    a.y = __fadd_rn(a.y, __fmul_rn(dt, b.y));
    a.z = __fadd_rn(a.z, __fmul_rn(dt, b.z));
    a.w = __fadd_rn(a.w, __fmul_rn(dt, b.w));
    __stcs(x4 + i, a);
  }
  // scalar tail (n not a multiple of 4)
  const long long t = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n && t < (n4 << 2) + 4) x[t] = __fadd_rn(x[t], __fmul_rn(dt, v[t]));
}

// -------------------------------------------------------------------- GEMV
// y[o] = sum_k W[o, k] act(x[k]) + b[o], W bf16 [O, K]; act = SiLU or none.
// The input vector is staged once per block in shared memory; each warp
// streams whole weight rows with 16-byte loads.
constexpr int GEMV_ROWS_PER_WARP = 4;

__global__ void __launch_bounds__(256) gemv_kernel(const __nv_bfloat16* __restrict__ W,
                                                   const float* __restrict__ x,
                                                   const float* __restrict__ b,
                                                   float* __restrict__ y, int O, int K,
                                                   int silu_in) {
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ float xs[];
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const float t = x[k];
    xs[k] = silu_in ? t / (1.0f + expf(-t)) : t;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int k8 = K >> 3;
  for (int rr = 0; rr < GEMV_ROWS_PER_WARP; ++rr) {
    const int o = (blockIdx.x * nw + warp) * GEMV_ROWS_PER_WARP + rr;
    if (o >= O) break;
    const uint4* wr = reinterpret_cast<const uint4*>(W + (size_t)o * K);
    float acc = 0.f;
    for (int i = lane; i < k8; i += 32) {
      const uint4 u = __ldcs(wr + i);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
      const float* xv = xs + i * 8;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        acc = fmaf(f.x, xv[2 * e], acc);
        acc = fmaf(f.y, xv[2 * e + 1], acc);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) y[o] = acc + (b ? b[o] : 0.0f);
  }
}

// ---------------------------------------------------------------- sinusoid
// e = [cos(T w_j), sin(T w_j)], w_j = 10000^(-j / half), cosine half first
// ([ZFLOW] section IV: flip_sin_to_cos).
__global__ void sinusoid_kernel(float T, int dim, float* out) {
  grid_dep_wait();
  grid_dep_launch();
  const int half = dim / 2;
  for (int j = threadIdx.x; j < half; j += blockDim.x) {
    const float w = (float)exp(-log(10000.0) * (double)j / (double)half);
    const float arg = T * w;
    out[j] = cosf(arg);
    out[half + j] = sinf(arg);
  }
}

// -------------------------------------------------------------- RoPE tables
// Multi-axis RoPE ([ERNIE] section I: axes [32,48,48], theta 256; section IV
// token layout; section VII, Decision 3).  Pair k of the head vector belongs
// to axis a when it falls in that axis's chunk; it turns by
// pos_a * theta^(-2 j / axes[a]) (j = pair index inside the chunk), the
// frequency rounded to float from double, the product in float.  Tables are
// pair-major, [d/2][n]: the QKV epilogue holds one token per lane, so a warp
// reads 32 consecutive tokens of one pair in one coalesced request.
struct Axes3 {
  int a0, a1, a2;
};

__global__ void rope_grid_kernel(int grid_h, int grid_w, int n_txt, const int* __restrict__ pos,
                                 int n, Axes3 axes, float theta, int half_d,
                                 float* __restrict__ cos_out, float* __restrict__ sin_out) {
  grid_dep_wait();
  grid_dep_launch();
  const long long total = (long long)n * half_d;
  const int n_img = grid_h * grid_w;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i / n);
    const int t = (int)(i - (long long)k * n);
    int p0, p1, p2;
    if (pos) {
      p0 = pos[3 * t];
      p1 = pos[3 * t + 1];
      p2 = pos[3 * t + 2];
    } else if (t < n_img) {
      p0 = n_txt;
      p1 = t / grid_w;
      p2 = t % grid_w;
    } else {
      p0 = t - n_img;
      p1 = 0;
      p2 = 0;
    }
    int axis_size, j, p;
    if (k < axes.a0 / 2) {
      axis_size = axes.a0; j = k; p = p0;
    } else if (k < axes.a0 / 2 + axes.a1 / 2) {
      axis_size = axes.a1; j = k - axes.a0 / 2; p = p1;
    } else {
      axis_size = axes.a2; j = k - axes.a0 / 2 - axes.a1 / 2; p = p2;
    }
    const float inv = (float)pow((double)theta, -2.0 * (double)j / (double)axis_size);
    const float ang = (float)p * inv;
    cos_out[i] = cosf(ang);
    sin_out[i] = sinf(ang);
  }
}

// Rotate-half tables of the pre-norm ViT: prefix tokens unrotated, patch
// (r, c): pair k < d/4 turns by r w_k, pair d/4 + k by c w_k,
// w_k = base^(-k / (d/4)).  Pair-major like the grid tables.
__global__ void rope_vit_kernel(int grid_h, int grid_w, int n_prefix, int head_dim, float base,
                                float* __restrict__ cos_out, float* __restrict__ sin_out) {
  grid_dep_wait();
  grid_dep_launch();
  const int half = head_dim / 2, q = head_dim / 4;
  const long long n = (long long)n_prefix + (long long)grid_h * grid_w;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n * half;
       i += (long long)gridDim.x * blockDim.x) {
    const int k = (int)(i / n);
    const int t = (int)(i - (long long)k * n);
    float ang = 0.0f;
    if (t >= n_prefix) {
      const int pidx = t - n_prefix;
      const int r = pidx / grid_w, c = pidx % grid_w;
      const int kk = k < q ? k : k - q;
      const float w = (float)pow((double)base, -(double)kk / (double)q);
      ang = (float)(k < q ? r : c) * w;
    }
    cos_out[i] = cosf(ang);
    sin_out[i] = sinf(ang);
  }
}

// ------------------------------------------------------------------- casts
__global__ void f32_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                   long long n) {
  grid_dep_wait();
  grid_dep_launch();
  const long long n4 = n >> 2;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 f = reinterpret_cast<const float4*>(in)[i];
    uint2 u;
    u.x = pack_bf16x2(f.x, f.y);
    u.y = pack_bf16x2(f.z, f.w);
    reinterpret_cast<uint2*>(out)[i] = u;
  }
  const long long t = (n4 << 2) + (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n && t < (n4 << 2) + 4) out[t] = __float2bfloat16_rn(in[t]);
}

// hi = bf16(x), lo = bf16(x - hi): x to about 16 significant bits as two
// bf16 operands.
__global__ void split_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ hi,
                                  __nv_bfloat16* __restrict__ lo, long long n) {
  grid_dep_wait();
  grid_dep_launch();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float x = in[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
  }
}

__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ in, float* __restrict__ out,
                                   long long n) {
  grid_dep_wait();
  grid_dep_launch();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    out[i] = __bfloat162float(in[i]);
}

// A wait that nothing completes: exercises the bounded-wait failure path.
__global__ void stuck_wait_kernel(DevErr e) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, e);
}

inline int grid_for(long long work, int threads, int sm_count) {
  long long g = (work + threads - 1) / threads;
  const long long cap = (long long)sm_count * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_ln_modulate(int mode, const float* x, long long ldx, int rows, int H,
                               const float* p0, const float* p1, float eps,
                               __nv_bfloat16* out, long long ldo, cudaStream_t st,
                               __nv_bfloat16* out_lo) {
  if (H > LN_THREADS * 4 * LN_MAXV || (H & 3)) return cudaErrorInvalidValue;
  const int grid = rows;
  if (grid == 0) return cudaSuccess;
  // widths the warp-per-row kernel is built for
  if (H == 1024 || H == 256) {
    const int g = (rows + LNW_WARPS - 1) / LNW_WARPS;
#define DIT_LNW(M, R, NV)                                                                    \
  launch_k(ln_modulate_warp_kernel<M, R, NV>, dim3(g), dim3(LNW_WARPS * 32), 0, st, 1, x, ldx, \
           rows, p0, p1, eps, out, ldo, out_lo)
#define DIT_LNW_H(M, R) return (H == 1024 ? DIT_LNW(M, R, 8) : DIT_LNW(M, R, 2))
    switch (mode) {
      case 0: DIT_LNW_H(0, false);
      case 1: DIT_LNW_H(1, false);
      case 2: DIT_LNW_H(0, true);
      case 3: DIT_LNW_H(1, true);
      default: return cudaErrorInvalidValue;
    }
#undef DIT_LNW_H
#undef DIT_LNW
  }
  const bool small = H <= LN_THREADS * 4 * 4;
#define DIT_LN_LAUNCH(M, R)                                                                  \
  return small ? launch_k(ln_modulate_kernel<M, R, 4>, dim3(grid), dim3(LN_THREADS), 0, st, 1, \
                          x, ldx, rows, H, p0, p1, eps, out, ldo, out_lo)                   \
               : launch_k(ln_modulate_kernel<M, R, LN_MAXV>, dim3(grid), dim3(LN_THREADS), 0,  \
                          st, 1, x, ldx, rows, H, p0, p1, eps, out, ldo, out_lo)
  switch (mode) {
    case 0: DIT_LN_LAUNCH(0, false);
    case 1: DIT_LN_LAUNCH(1, false);
    case 2: DIT_LN_LAUNCH(0, true);
    case 3: DIT_LN_LAUNCH(1, true);
    default: return cudaErrorInvalidValue;
  }
#undef DIT_LN_LAUNCH
}

cudaError_t launch_euler(float* x, const float* v, long long n, float dt, cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  if (n == 0) return cudaSuccess;
  return launch_k(euler_kernel, dim3(grid_for((n + 3) / 4, 256, ds->sm_count)), dim3(256), 0, st,
                  1, x, v, n, dt);
}

cudaError_t launch_gemv(const __nv_bfloat16* W, const float* x, const float* b, float* y, int O,
                        int K, int silu_in, cudaStream_t st) {
  if ((K & 7) || K > GEMV_MAX_K) return cudaErrorInvalidValue;
  const int rows_per_block = 8 * GEMV_ROWS_PER_WARP;
  const int grid = (O + rows_per_block - 1) / rows_per_block;
  const size_t smem = (size_t)K * sizeof(float);
  if (smem > 48 * 1024) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           GEMV_MAX_K * (int)sizeof(float));
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  return launch_k(gemv_kernel, dim3(grid), dim3(256), smem, st, 1, W, x, b, y, O, K, silu_in);
}

cudaError_t launch_sinusoid(float T, int dim, float* out, cudaStream_t st) {
  return launch_k(sinusoid_kernel, dim3(1), dim3(128), 0, st, 1, T, dim, out);
}

cudaError_t launch_rope_grid(int grid_h, int grid_w, int n_txt, const int* pos, int n_pos,
                             const int32_t* axes, float theta, int half_d, float* cos_out,
                             float* sin_out, cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  const int n = pos ? n_pos : grid_h * grid_w + n_txt;
  const long long total = (long long)n * half_d;
  if (total == 0) return cudaSuccess;
  return launch_k(rope_grid_kernel, dim3(grid_for(total, 256, ds->sm_count)), dim3(256), 0, st, 1,
                  grid_h, grid_w, n_txt, pos, n, Axes3{axes[0], axes[1], axes[2]}, theta, half_d,
                  cos_out, sin_out);
}

cudaError_t launch_rope_vit(int grid_h, int grid_w, int n_prefix, int head_dim, float base,
                            float* cos_out, float* sin_out, cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  const long long total = ((long long)n_prefix + (long long)grid_h * grid_w) * (head_dim / 2);
  if (total == 0) return cudaSuccess;
  return launch_k(rope_vit_kernel, dim3(grid_for(total, 256, ds->sm_count)), dim3(256), 0, st, 1,
                  grid_h, grid_w, n_prefix, head_dim, base, cos_out, sin_out);
}

cudaError_t launch_f32_to_bf16(const float* in, __nv_bfloat16* out, long long n, cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  if (n == 0) return cudaSuccess;
  return launch_k(f32_to_bf16_kernel, dim3(grid_for((n + 3) / 4, 256, ds->sm_count)), dim3(256),
                  0, st, 1, in, out, n);
}

cudaError_t launch_split_bf16(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, long long n,
                              cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  if (n == 0) return cudaSuccess;
  return launch_k(split_bf16_kernel, dim3(grid_for(n, 256, ds->sm_count)), dim3(256), 0, st, 1,
                  in, hi, lo, n);
}

cudaError_t launch_bf16_to_f32(const __nv_bfloat16* in, float* out, long long n, cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  if (n == 0) return cudaSuccess;
  return launch_k(bf16_to_f32_kernel, dim3(grid_for(n, 256, ds->sm_count)), dim3(256), 0, st, 1,
                  in, out, n);
}

cudaError_t launch_stuck_wait(DevErr e, cudaStream_t st) {
  return launch_k(stuck_wait_kernel, dim3(1), dim3(32), 0, st, 1, e);
}

}  // namespace dit
