// Persistent, warp-specialised tcgen05 GEMM with fused epilogues (the kernel
// template; gemm.cu launches the bf16 instances, gemm_f8.cu the e4m3 ones).
//
// D[M, N] = A[M, K] B[N, K]^T: bf16 operands staged in shared memory by TMA
// (128-byte swizzle), 128 x 256 x 64 tiles, fp32 accumulators in tensor
// memory, double-buffered so that the epilogue of one tile overlaps the
// main loop of the next.  Roles per CTA (192 threads, one CTA per SM):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator and MMA issuer (one lane)
//   warps 2..5  epilogue: thread t of the group owns accumulator row t
//
// The epilogues are the fused pointwise tails of the block's linears
// ([ZFLOW] "From Python + CUDA to Pure Rust + Metal 4", section VI: fused
// epilogues GatedResidual, Glu; [ERNIE] "Porting ERNIE-Image-Turbo to Zig and
// Metal", section IV per-layer graph and section VII, Decision 1: fp32
// residual):
//   EPI_BF16      plain bf16 store
//   EPI_F32_BIAS  fp32 store with bias (patch embedding, output projection)
//   EPI_RESIDUAL  x += gate * y on the fp32 residual stream (out, down)
//   EPI_SWIGLU    h = SiLU(gate) * up, gate and up columns in one tile
//   EPI_GEGLU     the same with the clamped tanh GELU ([ERNIE] section V, Bug 1)
//   EPI_RESIDUAL_TANH / _SIGMOID  x += f(gate) * y ([ZFLOW] sections IV, V)
//   EPI_QKV       per-head LayerNorm of q and k with gain/bias, then RoPE;
//                 q and k written head-major, v transposed per sequence, the
//                 layouts the attention kernel loads as contiguous tiles
//
// With F8 the operands are e4m3 codes with one fp32 scale per row of A and per
// row of B, the per-row 8-bit format of [ZFLOW] section VII; the epilogue
// first multiplies each accumulator by its two scales, then runs as above.
#pragma once

#include "internal.h"

namespace dit {
namespace {

// One pipeline stage holds 128 bytes of K per operand row: 64 bf16 or 128
// e4m3 values, the same 128-byte swizzled layout either way.
constexpr int BM = 128, BN = 256, BK_BYTES = 128, STAGES = 4;
constexpr int A_BYTES = BM * BK_BYTES;
constexpr int B_BYTES = BN * BK_BYTES;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_THREADS = 192;

struct GemmBars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_slot;
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024 + sizeof(GemmBars) + 64;

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d[q] = u;
  }
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// GELU by its tanh approximation, the argument limited to [-20, 20] and the
// result to [-65504, 65504] ([ERNIE] section V, Bug 1).
__device__ __forceinline__ float gelu_tanh_clamped_f(float x) {
  float a = 0.7978845608f * (x + 0.044715f * x * x * x);
  a = fminf(fmaxf(a, -20.0f), 20.0f);
  const float y = 0.5f * x * (1.0f + tanhf(a));
  return fminf(fmaxf(y, -65504.0f), 65504.0f);
}

// The gate function of a gated residual: identity, tanh or sigmoid.
template <int EPI>
__device__ __forceinline__ float gate_f(float g) {
  if constexpr (EPI == EPI_RESIDUAL_TANH) return tanhf(g);
  if constexpr (EPI == EPI_RESIDUAL_SIGMOID) return 1.0f / (1.0f + expf(-g));
  return g;
}

template <int EPI>
constexpr bool is_residual() {
  return EPI == EPI_RESIDUAL || EPI == EPI_RESIDUAL_TANH || EPI == EPI_RESIDUAL_SIGMOID;
}

// Rotates the pairs of one head row by the RoPE table row of its token:
// pairs (2k, 2k+1) or (k, k + HD/2), angle k.
template <int HD>
__device__ __forceinline__ void rope_row(float (&v)[HD], const QkvEpi& q, int row) {
  const int trow = row % q.s_len;
  const float4* cs = reinterpret_cast<const float4*>(q.rcos + (size_t)trow * (HD / 2));
  const float4* sn = reinterpret_cast<const float4*>(q.rsin + (size_t)trow * (HD / 2));
#pragma unroll
  for (int k4 = 0; k4 < HD / 8; ++k4) {
    const float4 c4 = __ldg(cs + k4), s4 = __ldg(sn + k4);
    const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
    const float ssn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 4 * k4 + e;
      if (q.rope_half) {
        const float a = v[k], bb = v[k + HD / 2];
        v[k] = a * cc[e] - bb * ssn[e];
        v[k + HD / 2] = a * ssn[e] + bb * cc[e];
      } else {
        const float a = v[2 * k], bb = v[2 * k + 1];
        v[2 * k] = a * cc[e] - bb * ssn[e];
        v[2 * k + 1] = a * ssn[e] + bb * cc[e];
      }
    }
  }
}

// Multiplies 32 accumulator columns starting at `col` by the row scale and
// the columns' scales (columns at or past n are left alone).
__device__ __forceinline__ void scale_cols(float (&v)[32], float rs, const float* sb, int col,
                                           int n) {
  if (col + 32 <= n) {
    const float4* s4 = reinterpret_cast<const float4*>(sb + col);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 s = __ldg(s4 + q);
      v[4 * q + 0] *= rs * s.x;
      v[4 * q + 1] *= rs * s.y;
      v[4 * q + 2] *= rs * s.z;
      v[4 * q + 3] *= rs * s.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col + i < n) v[i] *= rs * __ldg(sb + col + i);
  }
}

// ---------------------------------------------------------------- epilogues
template <int EPI, int HD, bool F8>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t tbase, int row,
                                              int n_blk) {
  const bool row_ok = row < p.M;
  float rs = 1.0f;
  if constexpr (F8) rs = row_ok ? __ldg(p.sa + row) : 0.0f;
  if constexpr (EPI == EPI_BF16 || EPI == EPI_F32_BIAS || is_residual<EPI>()) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col = n_blk * BN + c * 32;
      if (col >= p.N) break;
      float v[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, v);
      if (!row_ok) continue;  // the loads above stay warp-uniform
      if constexpr (F8) scale_cols(v, rs, p.sb, col, p.N);
      const bool full = col + 32 <= p.N;
      if constexpr (EPI == EPI_BF16) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.ldo + col;
        if (full) {
          store_bf16x32(dst, v);
        } else {
          for (int i = 0; i < 32 && col + i < p.N; ++i) dst[i] = __float2bfloat16_rn(v[i]);
        }
      } else if constexpr (EPI == EPI_F32_BIAS) {
        float* dst = reinterpret_cast<float*>(p.out) + (size_t)row * p.ldo + col;
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 o;
            o.x = v[4 * q + 0];
            o.y = v[4 * q + 1];
            o.z = v[4 * q + 2];
            o.w = v[4 * q + 3];
            if (p.vec) {
              const float4 b = __ldg(reinterpret_cast<const float4*>(p.vec + col) + q);
              o.x += b.x; o.y += b.y; o.z += b.z; o.w += b.w;
            }
            reinterpret_cast<float4*>(dst)[q] = o;
          }
        } else {
          for (int i = 0; i < 32 && col + i < p.N; ++i)
            dst[i] = v[i] + (p.vec ? __ldg(p.vec + col + i) : 0.0f);
        }
      } else {  // gated residual
        float* dst = reinterpret_cast<float*>(p.out) + (size_t)row * p.ldo + col;
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 x = reinterpret_cast<float4*>(dst)[q];
            float4 g = make_float4(1.f, 1.f, 1.f, 1.f);
            if (p.vec) {
              g = __ldg(reinterpret_cast<const float4*>(p.vec + col) + q);
              g.x = gate_f<EPI>(g.x);
              g.y = gate_f<EPI>(g.y);
              g.z = gate_f<EPI>(g.z);
              g.w = gate_f<EPI>(g.w);
            }
            x.x = fmaf(g.x, v[4 * q + 0], x.x);
            x.y = fmaf(g.y, v[4 * q + 1], x.y);
            x.z = fmaf(g.z, v[4 * q + 2], x.z);
            x.w = fmaf(g.w, v[4 * q + 3], x.w);
            reinterpret_cast<float4*>(dst)[q] = x;
          }
        } else {
          for (int i = 0; i < 32 && col + i < p.N; ++i)
            dst[i] = fmaf(p.vec ? gate_f<EPI>(__ldg(p.vec + col + i)) : 1.0f, v[i], dst[i]);
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GEGLU) {
    // Accumulator columns [0, 128) are gate rows, [128, 256) the matching up rows.
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float g[32], u[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, g);
      tmem_ld32(tbase + 128 + c * 32, u);
      if (!row_ok) continue;
      if constexpr (F8) {  // gate rows' scales first, then the up rows'
        scale_cols(g, rs, p.sb, n_blk * 128 + c * 32, p.N);
        scale_cols(u, rs, p.sb + p.N, n_blk * 128 + c * 32, p.N);
      }
      if constexpr (EPI == EPI_GEGLU) {
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] = gelu_tanh_clamped_f(g[i]) * u[i];
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
      }
      __nv_bfloat16* dst =
          reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.ldo + n_blk * 128 + c * 32;
      store_bf16x32(dst, g);
    }
  } else if constexpr (EPI == EPI_QKV) {
    const QkvEpi& q = p.qkv;
    constexpr int HPT = BN / HD;  // heads per tile
#pragma unroll 1
    for (int hh = 0; hh < HPT; ++hh) {
      const int col0 = n_blk * BN + hh * HD;
      if (col0 >= p.N) break;
      const int head = col0 / HD;
      float v[HD];
      __syncwarp();
#pragma unroll
      for (int c = 0; c < HD / 32; ++c)
        tmem_ld32(tbase + hh * HD + c * 32, *reinterpret_cast<float(*)[32]>(&v[c * 32]));
      if (!row_ok) continue;
      if constexpr (F8) {
#pragma unroll
        for (int c = 0; c < HD / 32; ++c)
          scale_cols(*reinterpret_cast<float(*)[32]>(&v[c * 32]), rs, p.sb, col0 + c * 32, p.N);
      }
      if (head < q.nh + q.nkv) {
        const bool is_q = head < q.nh;
        const float* g = is_q ? q.qg : q.kg;
        const float* b = is_q ? q.qb : q.kb;
        if (q.rope_first) rope_row<HD>(v, q, row);
        if (g != nullptr) {
          // per-head LayerNorm or RMSNorm over the head_dim values of this row
          float mean = 0.f;
          if (!q.rms) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < HD; ++i) s += v[i];
            mean = s * (1.0f / HD);
          }
          float ss = 0.f;
#pragma unroll
          for (int i = 0; i < HD; ++i) {
            v[i] -= mean;
            ss = fmaf(v[i], v[i], ss);
          }
          const float rstd = 1.0f / sqrtf(ss * (1.0f / HD) + q.eps);
#pragma unroll
          for (int i = 0; i < HD; ++i) v[i] = fmaf(v[i] * rstd, __ldg(g + i), __ldg(b + i));
        }
        if (!q.rope_first) rope_row<HD>(v, q, row);
        // head-major: one head's rows are contiguous, so an attention tile of
        // 128 tokens x d is one contiguous block
        __nv_bfloat16* dst = q.qk + ((size_t)head * p.M + row) * HD;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c)
          store_bf16x32(dst + c * 32, *reinterpret_cast<float(*)[32]>(&v[c * 32]));
      } else {
        const int g = head - q.nh - q.nkv;
        const int seq = row / q.s_len;
        const int j = row - seq * q.s_len;
        __nv_bfloat16* dst = q.vt + ((size_t)(seq * q.nkv + g) * HD) * q.s_pad + j;
#pragma unroll
        for (int c = 0; c < HD; ++c) dst[(size_t)c * q.s_pad] = __float2bfloat16_rn(v[c]);
      }
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int EPI, int HD, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + (size_t)STAGES * STAGE_BYTES);

  const int warp = warp_id(), lane = lane_id();
  const int num_tiles = p.num_m * p.num_n;
  constexpr int BK = F8 ? BK_BYTES : BK_BYTES / 2;  // K elements per stage
  const int k_blocks = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 4);
    }
    mbar_init(&bars->drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        const int m_blk = t % p.num_m, n_blk = t / p.num_m;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          mbar_arrive_expect_tx(&bars->full[stage], STAGE_BYTES);
          tma_load_2d(sa, &tmA, &bars->full[stage], kb * BK, m_blk * BM);
          if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GEGLU) {
            tma_load_2d(sb, &tmB, &bars->full[stage], kb * BK, n_blk * 128);
            tma_load_2d(sb + B_BYTES / 2, &tmB, &bars->full[stage], kb * BK, p.N + n_blk * 128);
          } else {
            tma_load_2d(sb, &tmB, &bars->full[stage], kb * BK, n_blk * BN);
          }
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy issued must have landed before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if (filled & (1u << s)) mbar_wait(&bars->full[s], (fill_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + (size_t)stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
          // four MMAs per stage, each over 32 bytes of K (16 bf16 or 32 e4m3)
#pragma unroll
          for (int k = 0; k < BK_BYTES / 32; ++k) {
            if constexpr (F8)
              umma_e4m3(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32),
                        idesc, (kb | k) != 0);
            else
              umma_bf16(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32),
                        idesc, (kb | k) != 0);
          }
          umma_commit(&bars->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&bars->tfull[acc]);
      }
      // All MMAs issued must complete before TMEM is released.
      umma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.err);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int quarter = warp & 3;  // TMEM lanes [32 quarter, 32 quarter + 32)
    const int r_in = quarter * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
      const int m_blk = t % p.num_m, n_blk = t / p.num_m;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(&bars->tfull[acc], acc_phase, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
      epilogue_tile<EPI, HD, F8>(p, tbase, m_blk * BM + r_in, n_blk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int EPI, int HD, bool F8>
cudaError_t launch_impl(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                        int grid, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<EPI, HD, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  gemm_kernel<EPI, HD, F8><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ta, tb, p);
  count_launch();
  return cudaGetLastError();
}

// Encodes the two operand maps (boxes of 128 bytes of K by 128 or 256 rows),
// counts the tiles and launches one persistent CTA per SM at most.
template <bool F8>
cudaError_t launch_gemm_t(int epi, int hd, const void* A, long long lda, const void* B,
                          long long ldb, GemmParams& p, cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  constexpr uint32_t ES = F8 ? 1 : 2;
  constexpr uint32_t BK = BK_BYTES / ES;
  CUtensorMap ta, tb;
  {
    const uint64_t dims[2] = {(uint64_t)p.K, (uint64_t)p.M};
    const uint64_t strides[1] = {(uint64_t)lda * ES};
    const uint32_t box[2] = {BK, BM};
    if (!make_tmap(&ta, ES, A, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const bool glu = epi == EPI_SWIGLU || epi == EPI_GEGLU;
  {
    const uint64_t rows = glu ? 2ull * p.N : (uint64_t)p.N;
    const uint64_t dims[2] = {(uint64_t)p.K, rows};
    const uint64_t strides[1] = {(uint64_t)ldb * ES};
    const uint32_t box[2] = {BK, glu ? 128u : (uint32_t)BN};
    if (!make_tmap(&tb, ES, B, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  p.num_m = (p.M + BM - 1) / BM;
  p.num_n = glu ? p.N / 128 : (p.N + BN - 1) / BN;
  p.err = dev_err(ds);
  const int tiles = p.num_m * p.num_n;
  const int grid = tiles < ds->sm_count ? tiles : ds->sm_count;
  switch (epi) {
    case EPI_BF16: return launch_impl<EPI_BF16, 0, F8>(ta, tb, p, grid, st);
    case EPI_F32_BIAS: return launch_impl<EPI_F32_BIAS, 0, F8>(ta, tb, p, grid, st);
    case EPI_RESIDUAL: return launch_impl<EPI_RESIDUAL, 0, F8>(ta, tb, p, grid, st);
    case EPI_SWIGLU: return launch_impl<EPI_SWIGLU, 0, F8>(ta, tb, p, grid, st);
    case EPI_GEGLU: return launch_impl<EPI_GEGLU, 0, F8>(ta, tb, p, grid, st);
    case EPI_RESIDUAL_TANH: return launch_impl<EPI_RESIDUAL_TANH, 0, F8>(ta, tb, p, grid, st);
    case EPI_RESIDUAL_SIGMOID:
      return launch_impl<EPI_RESIDUAL_SIGMOID, 0, F8>(ta, tb, p, grid, st);
    case EPI_QKV:
      if (hd == 64) return launch_impl<EPI_QKV, 64, F8>(ta, tb, p, grid, st);
      if (hd == 128) return launch_impl<EPI_QKV, 128, F8>(ta, tb, p, grid, st);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace dit
