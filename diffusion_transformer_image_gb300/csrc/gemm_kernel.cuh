// Persistent, warp-specialised tcgen05 GEMM with fused epilogues (the kernel
// template; gemm.cu launches the bf16 instances, gemm_f8.cu the e4m3 ones).
//
// D[M, N] = A[M, K] B[N, K]^T: bf16 operands staged in shared memory by TMA
// (128-byte swizzle), fp32 accumulators in tensor memory, double-buffered so
// that the epilogue of one tile overlaps the main loop of the next.  A cluster
// of two CTAs (on two SMs) computes one 256 x 256 tile with tcgen05 pair MMAs
// (cta_group::2): each CTA stages its 128 rows of A and 128 of the tile's 256
// rows of B, 64 values of K per stage, so a stage is 32 KB per SM (a single
// CTA's 128 x 256 tile would need 48 KB for the same MMA work per SM) and six
// stages fit.  Rank 0 of the pair issues the MMAs for both; each CTA's tensor
// memory holds the 128 accumulator rows of its half.  Roles per CTA (192
// threads, one CTA per SM):
//   warp 0      TMA producer (one lane); both CTAs' copies complete on rank 0's
//               stage barrier
//   warp 1      TMEM allocator (both CTAs) and MMA issuer (one lane of rank 0)
//   warps 2..5  epilogue: thread t of the group owns accumulator row t of its
//               CTA's half
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
//   EPI_EULER     the second (low-half) pass of the output projection: the
//                 velocity v = out + y is completed and the flow-matching Euler
//                 update latent += (sigma_next - sigma) v applied, the product
//                 rounded before the add ([ZFLOW] section IV, Euler sign +1)
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
// e4m3 values, the same 128-byte swizzled layout either way.  BM rows of A
// and BNH rows of B per CTA; PM x BN output rows x columns per CTA pair.
constexpr int BM = 128, BN = 256, BK_BYTES = 128, STAGES = 6;
constexpr int PM = 2 * BM;
constexpr int BNH = BN / 2;
constexpr int A_BYTES = BM * BK_BYTES;
constexpr int B_BYTES = BNH * BK_BYTES;
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

// Epilogue staging: each epilogue warp owns two buffers of 32 rows x 128
// bytes (its TMEM lane quarter x one chunk of columns) in the 128-byte
// swizzled layout, written by the threads and stored to global memory by TMA.
constexpr int EBUF_BYTES = 32 * 128;
constexpr int EPI_SMEM = 4 * 2 * EBUF_BYTES;

// Epilogues that stage their output (the others keep that shared memory as L1
// for their table and parameter loads).
template <int EPI>
constexpr bool is_staged() {
  return EPI == EPI_BF16 || EPI == EPI_SWIGLU || EPI == EPI_GEGLU || EPI == EPI_RESIDUAL ||
         EPI == EPI_RESIDUAL_TANH || EPI == EPI_RESIDUAL_SIGMOID || EPI == EPI_QKV;
}
template <int EPI>
constexpr size_t smem_bytes() {
  return (size_t)STAGES * STAGE_BYTES + (is_staged<EPI>() ? EPI_SMEM : 0) + 1024 +
         sizeof(GemmBars) + 64;
}
static_assert(smem_bytes<EPI_RESIDUAL>() <= 232448, "shared memory per CTA exceeded");

// One epilogue warp's staging buffers and which one is next.
struct EpiStage {
  uint8_t* buf;
  int cur;
};

// Next staging buffer of this warp, once the TMA operation that read it two
// chunks ago has finished reading.
__device__ __forceinline__ uint8_t* ebuf_acquire(EpiStage& es, int lane) {
  if (lane == 0) bulk_wait_read<1>();
  __syncwarp();
  return es.buf + es.cur * EBUF_BYTES;
}

// Makes the warp's stores to the buffer visible to the TMA unit; lane 0 then
// issues the store and commits it.
__device__ __forceinline__ void ebuf_release(EpiStage& es) {
  fence_proxy_async_smem();
  __syncwarp();
  es.cur ^= 1;
}

// 16 bytes into row r, piece j (0..7) of a swizzled staging buffer.
__device__ __forceinline__ void ebuf_put16(uint8_t* b, int r, int j, uint4 v) {
  *reinterpret_cast<uint4*>(b + r * 128 + ((j ^ (r & 7)) << 4)) = v;
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

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

// SiLU with the hardware exponential and a fast divide: relative error a few
// fp32 ulps, far below the bf16 output's resolution.
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

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

// Loads kept in program order (volatile asm) so that a request stays ahead of
// the TMEM reads whose latency it is meant to overlap; the tcgen05.ld
// wrappers are compiler memory barriers, so plain loads would be issued only
// after them.  The RoPE tables stream through without allocating in L1 (they
// would evict the gains, biases and column scales that every warp reads).
__device__ __forceinline__ float ldg_stream(const float* p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ldg_ordered(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// The 16 pairs j*16 .. j*16+15 of one head row as two arrays (first and
// second element of each pair): interleaved pairs (2k, 2k+1) come from the
// 32 columns from 32 j, rotate-half pairs (k, k + HD/2) from the 16 columns
// from 16 j and the 16 from HD/2 + 16 j.
template <int HD>
__device__ __forceinline__ void tmem_pairs(uint32_t hb, bool half, int j, float (&a)[16],
                                           float (&b)[16]) {
  if (half) {
    tmem_ld16(hb + 16 * j, a);
    tmem_ld16(hb + HD / 2 + 16 * j, b);
  } else {
    float x[32];
    tmem_ld32(hb + 32 * j, x);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      a[e] = x[2 * e];
      b[e] = x[2 * e + 1];
    }
  }
}

// The arithmetic below runs on f32x2 operands over two neighbouring pairs:
// A = (a[e], a[e+1]) and B = (b[e], b[e+1]), e even, half the instructions
// of the scalar form.
__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

// Shifted sums of the 16 pairs j for the norm statistics: s1 += x - x0,
// s2 += (x - x0)^2 (x0 broadcast in nx0 as -x0).
__device__ __forceinline__ void stat_pairs(const float (&a)[16], const float (&b)[16], float2 nx0,
                                           float2 (&s1)[2], float2 (&s2)[2]) {
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    const float2 da = __fadd2_rn(f2(a[e], a[e + 1]), nx0);
    const float2 db = __fadd2_rn(f2(b[e], b[e + 1]), nx0);
    s1[0] = __fadd2_rn(s1[0], da);
    s1[1] = __fadd2_rn(s1[1], db);
    s2[0] = __ffma2_rn(da, da, s2[0]);
    s2[1] = __ffma2_rn(db, db, s2[1]);
  }
}

// x rstd - mean rstd, then times g plus b, on the 16 pairs j; the gains and
// biases read four columns at a time as they are used.
template <int HD>
__device__ __forceinline__ void norm_pairs(float (&a)[16], float (&b)[16], const float* g,
                                           const float* bias, bool half, int j, float mean,
                                           float rstd) {
  const float2 r2 = f2(rstd, rstd);
  const float2 o2 = f2(-mean * rstd, -mean * rstd);
  if (half) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // pairs 4 i .. 4 i + 3: columns 16 j + 4 i and HD/2 + 16 j + 4 i
      const float4 ga = __ldg(reinterpret_cast<const float4*>(g + 16 * j) + i);
      const float4 ba = __ldg(reinterpret_cast<const float4*>(bias + 16 * j) + i);
      const float4 gb = __ldg(reinterpret_cast<const float4*>(g + HD / 2 + 16 * j) + i);
      const float4 bb = __ldg(reinterpret_cast<const float4*>(bias + HD / 2 + 16 * j) + i);
      float2 x = __ffma2_rn(f2(a[4 * i], a[4 * i + 1]), r2, o2);
      x = __ffma2_rn(x, f2(ga.x, ga.y), f2(ba.x, ba.y));
      a[4 * i] = x.x;
      a[4 * i + 1] = x.y;
      x = __ffma2_rn(f2(a[4 * i + 2], a[4 * i + 3]), r2, o2);
      x = __ffma2_rn(x, f2(ga.z, ga.w), f2(ba.z, ba.w));
      a[4 * i + 2] = x.x;
      a[4 * i + 3] = x.y;
      x = __ffma2_rn(f2(b[4 * i], b[4 * i + 1]), r2, o2);
      x = __ffma2_rn(x, f2(gb.x, gb.y), f2(bb.x, bb.y));
      b[4 * i] = x.x;
      b[4 * i + 1] = x.y;
      x = __ffma2_rn(f2(b[4 * i + 2], b[4 * i + 3]), r2, o2);
      x = __ffma2_rn(x, f2(gb.z, gb.w), f2(bb.z, bb.w));
      b[4 * i + 2] = x.x;
      b[4 * i + 3] = x.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // columns 32 j + 4 i .. + 3: pairs 2 i, 2 i + 1
      const float4 gg = __ldg(reinterpret_cast<const float4*>(g + 32 * j) + i);
      const float4 bb = __ldg(reinterpret_cast<const float4*>(bias + 32 * j) + i);
      float2 x = __ffma2_rn(f2(a[2 * i], a[2 * i + 1]), r2, o2);
      x = __ffma2_rn(x, f2(gg.x, gg.z), f2(bb.x, bb.z));
      a[2 * i] = x.x;
      a[2 * i + 1] = x.y;
      x = __ffma2_rn(f2(b[2 * i], b[2 * i + 1]), r2, o2);
      x = __ffma2_rn(x, f2(gg.y, gg.w), f2(bb.y, bb.w));
      b[2 * i] = x.x;
      b[2 * i + 1] = x.y;
    }
  }
}

// Rotates pairs 16 j .. 16 j + 15 by this lane's table entries:
// a' = a c - b s, b' = a s + b c.
template <int HD>
__device__ __forceinline__ void rotate_pairs(float (&a)[16], float (&b)[16],
                                             const float (&tc)[HD / 2], const float (&ts)[HD / 2],
                                             int j) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float c = tc[16 * j + e], sn = ts[16 * j + e];
    const float x = a[e], y = b[e];
    a[e] = x * c - y * sn;
    b[e] = x * sn + y * c;
  }
}

// Writes the 16 pairs j of a head row as bf16 into the staging buffers of
// the warp (buffer = 64-column box of the head, 128-byte swizzled rows).
template <int HD>
__device__ __forceinline__ void stage_pairs(uint8_t* buf, int lane, bool half, int j,
                                            const float (&a)[16], const float (&b)[16]) {
  if (half) {
    const int ca = 16 * j, cb = HD / 2 + 16 * j;
    uint8_t* ba = buf + (ca >> 6) * EBUF_BYTES;
    uint8_t* bb = buf + (cb >> 6) * EBUF_BYTES;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ebuf_put16(ba, lane, ((ca & 63) >> 3) + i, pack_bf16x8(a + 8 * i));
      ebuf_put16(bb, lane, ((cb & 63) >> 3) + i, pack_bf16x8(b + 8 * i));
    }
  } else {
    const int c0 = 32 * j;
    uint8_t* bx = buf + (c0 >> 6) * EBUF_BYTES;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = a[4 * i + e];
        x[2 * e + 1] = b[4 * i + e];
      }
      ebuf_put16(bx, lane, ((c0 & 63) >> 3) + i, pack_bf16x8(x));
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

// Output tile coordinates of tile t: groups of group_m row blocks, row blocks
// fastest inside a group, so the pairs working at one time share the A rows
// of their group (and B tiles) in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& m_blk, int& n_blk) {
  const int per_group = p.group_m * p.num_n;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int rows = min(p.group_m, p.num_m - first);
  const int idx = t - g * per_group;
  m_blk = first + idx % rows;
  n_blk = idx / rows;
}

// ---------------------------------------------------------------- epilogues
// row: this thread's output row; row0: the first row of its warp's slab.
template <int EPI, int HD, bool F8>
// tmO: the output map of the staged epilogues (q/k heads for EPI_QKV); tmV:
// the transposed v of EPI_QKV.
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const CUtensorMap* tmO,
                                              const CUtensorMap* tmV, EpiStage& es,
                                              uint32_t tbase, int row, int row0, int lane,
                                              int n_blk) {
  const bool row_ok = row < p.M;
  float rs = 1.0f;
  if constexpr (F8) rs = row_ok ? __ldg(p.sa + row) : 0.0f;
  if constexpr (is_residual<EPI>()) {
    // x += g y through the staging buffer and a TMA reduce-add: the add
    // happens in L2, the GEMM never reads x
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col = n_blk * BN + c * 32;
      if (col >= p.N) break;
      float v[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, v);
      if constexpr (F8) scale_cols(v, rs, p.sb, col, p.N);
      if (p.vec) {
        if (col + 32 <= p.N) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 g = __ldg(reinterpret_cast<const float4*>(p.vec + col) + q);
            v[4 * q + 0] *= gate_f<EPI>(g.x);
            v[4 * q + 1] *= gate_f<EPI>(g.y);
            v[4 * q + 2] *= gate_f<EPI>(g.z);
            v[4 * q + 3] *= gate_f<EPI>(g.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col + i < p.N) v[i] *= gate_f<EPI>(__ldg(p.vec + col + i));
        }
      }
      uint8_t* b = ebuf_acquire(es, lane);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        ebuf_put16(b, lane, q,
                   make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                              __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])));
      ebuf_release(es);
      if (lane == 0 && row0 < p.M) {  // a slab wholly below M stores nothing
        tma_reduce_add_2d(tmO, b, col, row0);
        bulk_commit();
      }
    }
  } else if constexpr (EPI == EPI_BF16) {
    // 64 columns (128 bytes of bf16) per staged chunk
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int col = n_blk * BN + c * 64;
      if (col >= p.N) break;
      float v[32], w[32];
      __syncwarp();
      tmem_ld32(tbase + c * 64, v);
      tmem_ld32(tbase + c * 64 + 32, w);
      if constexpr (F8) {
        scale_cols(v, rs, p.sb, col, p.N);
        scale_cols(w, rs, p.sb, col + 32, p.N);
      }
      uint8_t* b = ebuf_acquire(es, lane);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ebuf_put16(b, lane, q, pack_bf16x8(v + 8 * q));
        ebuf_put16(b, lane, 4 + q, pack_bf16x8(w + 8 * q));
      }
      ebuf_release(es);
      if (lane == 0 && row0 < p.M) {  // a slab wholly below M stores nothing
        tma_store_2d(tmO, b, col, row0);
        bulk_commit();
      }
    }
  } else if constexpr (EPI == EPI_F32_BIAS) {
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
    }
  } else if constexpr (EPI == EPI_EULER) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col = n_blk * BN + c * 32;
      if (col >= p.N) break;
      float v[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, v);
      if (!row_ok) continue;  // the loads above stay warp-uniform
      if constexpr (F8) scale_cols(v, rs, p.sb, col, p.N);
      float* vel = reinterpret_cast<float*>(p.out) + (size_t)row * p.ldo + col;
      float* lat = p.aux + (size_t)row * p.ldo + col;
      for (int i = 0; i < 32 && col + i < p.N; ++i) {
        const float vv = __fadd_rn(vel[i], v[i]);
        vel[i] = vv;
        lat[i] = __fadd_rn(lat[i], __fmul_rn(p.scalar, vv));
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GEGLU) {
    // Accumulator columns [0, 128) are gate rows, [128, 256) the matching up
    // rows; h leaves in two staged chunks of 64 columns.
#pragma unroll 1
    for (int c2 = 0; c2 < 2; ++c2) {
      uint8_t* b = nullptr;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int cc = c2 * 64 + half * 32;
        float g[32], u[32];
        __syncwarp();
        tmem_ld32(tbase + cc, g);
        tmem_ld32(tbase + 128 + cc, u);
        if constexpr (F8) {  // gate rows' scales first, then the up rows'
          scale_cols(g, rs, p.sb, n_blk * 128 + cc, p.N);
          scale_cols(u, rs, p.sb + p.N, n_blk * 128 + cc, p.N);
        }
        if constexpr (EPI == EPI_GEGLU) {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = gelu_tanh_clamped_f(g[i]) * u[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
        }
        if (half == 0) b = ebuf_acquire(es, lane);
#pragma unroll
        for (int q = 0; q < 4; ++q) ebuf_put16(b, lane, half * 4 + q, pack_bf16x8(g + 8 * q));
      }
      ebuf_release(es);
      if (lane == 0 && row0 < p.M) {  // a slab wholly below M stores nothing
        tma_store_2d(tmO, b, n_blk * 128 + c2 * 64, row0);
        bulk_commit();
      }
    }
  } else if constexpr (EPI == EPI_QKV) {
    const QkvEpi& q = p.qkv;
    constexpr int HPT = BN / HD;  // heads per tile
    constexpr int NCH = HD / 32;  // chunks of 32 columns (16 pairs) per head
    const int trow = row % q.s_len;
    // this lane's table entries for all HD/2 pairs, the same for every head
    // of the tile: requested once, before the first head's TMEM passes, so
    // that their latency overlaps them (tiles of v heads only skip them)
    float tc[HD / 2], ts[HD / 2];
    if ((n_blk * BN) / HD < q.nh + q.nkv) {
#pragma unroll
      for (int k = 0; k < HD / 2; ++k) {
        tc[k] = ldg_stream(q.rcos + (size_t)k * q.s_len + trow);
        ts[k] = ldg_stream(q.rsin + (size_t)k * q.s_len + trow);
      }
    }
#pragma unroll 1
    for (int hh = 0; hh < HPT; ++hh) {
      const int col0 = n_blk * BN + hh * HD;
      if (col0 >= p.N) break;
      const int head = col0 / HD;
      const uint32_t hb = tbase + hh * HD;   // this head's accumulator columns
      // W8A8: the head's column scales, lane l holding the one of column
      // 32 c + l (one coalesced load per 32 columns), passed to every lane by
      // a shuffle where a chunk is scaled
      float sbl[NCH];
      if constexpr (F8) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) sbl[c] = ldg_ordered(p.sb + col0 + 32 * c + lane);
      }
      __syncwarp();
      if (head < q.nh + q.nkv) {
        if constexpr (F8) {
          // the row and column scales applied once, in TMEM, so that every
          // later pass reads scaled values
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            float x[32];
            tmem_ld32(hb + 32 * c, x);
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] *= rs * __shfl_sync(0xffffffffu, sbl[c], i);
            tmem_st32(hb + 32 * c, x);
          }
        }
        const bool is_q = head < q.nh;
        const float* g = is_q ? q.qg : q.kg;
        const float* b = is_q ? q.qb : q.kb;
        // the norm statistics in one pass over TMEM (of the rotated row when
        // the rotation comes first): sums of x - x0 and of its squares, x0
        // the row's first value (a sample of the row, so the variance
        // formula does not cancel), four partial sums each
        float mean = 0.f, rstd = 1.f;
        if (g != nullptr) {
          float2 s1[2] = {f2(0.f, 0.f), f2(0.f, 0.f)}, s2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
          float x0 = 0.f;
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            float pa[16], pb[16];
            tmem_pairs<HD>(hb, q.rope_half, j, pa, pb);
            if (q.rope_first) rotate_pairs<HD>(pa, pb, tc, ts, j);
            if (j == 0 && !q.rms) x0 = pa[0];
            stat_pairs(pa, pb, f2(-x0, -x0), s1, s2);
          }
          const float m1 = ((s1[0].x + s1[0].y) + (s1[1].x + s1[1].y)) * (1.0f / HD);
          const float m2 = ((s2[0].x + s2[0].y) + (s2[1].x + s2[1].y)) * (1.0f / HD);
          // RMSNorm: x0 = 0 and no centring, m2 is the mean square
          mean = q.rms ? 0.0f : x0 + m1;
          const float var = q.rms ? m2 : fmaxf(m2 - m1 * m1, 0.0f);
          rstd = 1.0f / sqrtf(var + q.eps);
        }
        // chunk by chunk: norm and rotation in the block's order, bf16 into
        // the staging buffers (one per 64-column box); then one TMA box
        // (64, 32 rows) per 64 columns of the head-major map [head][token][d].
        // Rows past M are not written.
        if (lane == 0) bulk_wait_read<0>();   // both staging buffers free
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float pa[16], pb[16];
          tmem_pairs<HD>(hb, q.rope_half, j, pa, pb);
          if (q.rope_first) rotate_pairs<HD>(pa, pb, tc, ts, j);
          if (g != nullptr) norm_pairs<HD>(pa, pb, g, b, q.rope_half, j, mean, rstd);
          if (!q.rope_first) rotate_pairs<HD>(pa, pb, tc, ts, j);
          stage_pairs<HD>(es.buf, lane, q.rope_half, j, pa, pb);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < p.M) {  // a slab wholly below M stores nothing
#pragma unroll
          for (int c = 0; c < HD / 64; ++c)
            tma_store_3d(tmO, es.buf + c * EBUF_BYTES, c * 64, row0, head);
          bulk_commit();
        }
      } else {
        // v, transposed per sequence.  When the slab's existing rows (< M)
        // all lie in one sequence and start on a 16-byte boundary of the
        // transposed row, one TMA box (32 tokens x d channels) from a
        // transposed staging tile [d][32] that fills both staging buffers of
        // the warp; otherwise direct stores.
        const int g = head - q.nh - q.nkv;
        const int seq0 = row0 / q.s_len;
        const int j0 = row0 - seq0 * q.s_len;
        const int rows_end = min(row0 + 32, p.M);
        const bool staged = row0 < p.M && j0 % 8 == 0 && rows_end <= (seq0 + 1) * q.s_len;
        __nv_bfloat16* tb = reinterpret_cast<__nv_bfloat16*>(es.buf);
        if (staged && lane == 0) bulk_wait_read<0>();   // both staging buffers free
        __syncwarp();
        const int seq = row / q.s_len;
        __nv_bfloat16* dst =
            q.vt + ((size_t)(seq * q.nkv + g) * HD) * q.s_pad + (row - seq * q.s_len);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float x[32];
          tmem_ld32(hb + c * 32, x);
          if constexpr (F8) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] *= rs * __shfl_sync(0xffffffffu, sbl[c], i);
          }
          if (staged) {
#pragma unroll
            for (int i = 0; i < 32; ++i) tb[(c * 32 + i) * 32 + lane] = __float2bfloat16_rn(x[i]);
          } else if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              dst[(size_t)(c * 32 + i) * q.s_pad] = __float2bfloat16_rn(x[i]);
          }
        }
        if (staged) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(tmV, tb, j0, (seq0 * q.nkv + g) * HD);
            bulk_commit();
          }
        }
      }
      es.cur = 0;   // every staged write of this epilogue first waits for both buffers
    }
  }
}

// ---------------------------------------------------------------- kernel
template <int EPI, int HD, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmV,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + (size_t)STAGES * STAGE_BYTES +
                                               (is_staged<EPI>() ? EPI_SMEM : 0));

  const int warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_rank();  // 0 issues the pair's MMAs
  const int pair = (int)cluster_index(), num_pairs = (int)cluster_count();
  const int num_tiles = p.num_m * p.num_n;
  constexpr int BK = F8 ? BK_BYTES : BK_BYTES / 2;  // K elements per stage
  const int k_blocks = (p.K + BK - 1) / BK;

  // Barriers, the same layout in both CTAs.  Used on rank 0 only: full (both
  // CTAs' copies of a stage), tempty (both CTAs' epilogue warps), drain.
  // Used on both: empty and tfull, which rank 0's commits signal in both.
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->tfull[a], 1);
      mbar_init(&bars->tempty[a], 8);
    }
    mbar_init(&bars->drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&bars->tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;
  // With p.b_early the producer requests the B tiles of its first tile's
  // first stages (fresh stages: no empty wait) before the grid-dependency
  // wait, so that they load while the kernel before this one finishes.
  int b_pre = 0;
  if (p.b_early && warp == 0 && lane == 0) {
    int m_blk, n_blk;
    tile_coords(p, pair, m_blk, n_blk);
    const int b_row = (EPI == EPI_SWIGLU || EPI == EPI_GEGLU)
                          ? (rank ? p.N : 0) + n_blk * BNH
                          : n_blk * BN + (int)rank * BNH;
    b_pre = k_blocks < STAGES ? k_blocks : STAGES;
    for (int kb = 0; kb < b_pre; ++kb) {
      if (rank == 0) mbar_arrive_expect_tx(&bars->full[kb], 2 * STAGE_BYTES);
      tma_load_2d_pair(smem + (size_t)kb * STAGE_BYTES + A_BYTES, &tmB,
                       mapa_shared(smem_u32(&bars->full[kb]), 0), kb * BK, b_row);
    }
  }
  grid_dep_wait();  // the previous kernel's outputs (A, the residual x) are complete
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0, filled = 0, fill_parity = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs) {
        int m_blk, n_blk;
        tile_coords(p, t, m_blk, n_blk);
        const int a_row = m_blk * PM + (int)rank * BM;
        // GLU tiles: rank 0 stages the 128 gate rows, rank 1 the matching up rows
        const int b_row = (EPI == EPI_SWIGLU || EPI == EPI_GEGLU)
                              ? (rank ? p.N : 0) + n_blk * BNH
                              : n_blk * BN + (int)rank * BNH;
        for (int kb = 0; kb < k_blocks; ++kb) {
          // the first tile's first b_pre stages: B already requested
          const bool pre = t == pair && kb < b_pre;
          if (!pre && !mbar_wait(&bars->empty[stage], phase ^ 1u, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + (size_t)stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          if (rank == 0) {
            if (!pre) mbar_arrive_expect_tx(&bars->full[stage], 2 * STAGE_BYTES);
            filled |= 1u << stage;
            fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          }
          const uint32_t fb = mapa_shared(smem_u32(&bars->full[stage]), 0);
          tma_load_2d_pair(sa, &tmA, fb, kb * BK, a_row);
          if (!pre) tma_load_2d_pair(sb, &tmB, fb, kb * BK, b_row);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy issued must have landed before the CTAs may exit (rank 0's
      // stage barriers count both CTAs' copies).
      if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if (filled & (1u << s)) mbar_wait(&bars->full[s], (fill_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(PM, BN) : idesc_bf16_f32(PM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait_cluster(&bars->tempty[acc], acc_phase ^ 1u, p.err)) break;
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
              umma_e4m3_pair(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32),
                             idesc, (kb | k) != 0);
            else
              umma_bf16_pair(d_tmem, sdesc_sw128(a_addr + k * 32), sdesc_sw128(b_addr + k * 32),
                             idesc, (kb | k) != 0);
          }
          umma_commit_pair_both(&bars->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair_both(&bars->tfull[acc]);
      }
      // All MMAs issued must complete before TMEM is released.
      umma_commit_pair_self(&bars->drain);
      mbar_wait(&bars->drain, 0, p.err);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int quarter = warp & 3;  // TMEM lanes [32 quarter, 32 quarter + 32)
    const int r_in = quarter * 32 + lane;
    EpiStage es{smem + (size_t)STAGES * STAGE_BYTES + (size_t)quarter * 2 * EBUF_BYTES, 0};
    const uint32_t te0 = mapa_shared(smem_u32(&bars->tempty[0]), 0);  // rank 0's barriers
    const uint32_t te1 = mapa_shared(smem_u32(&bars->tempty[1]), 0);
    int local = 0;
    for (int t = pair; t < num_tiles; t += num_pairs, ++local) {
      int m_blk, n_blk;
      tile_coords(p, t, m_blk, n_blk);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(&bars->tfull[acc], acc_phase, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
      const int row_base = m_blk * PM + (int)rank * BM;
      epilogue_tile<EPI, HD, F8>(p, &tmO, &tmV, es, tbase, row_base + r_in,
                                 row_base + quarter * 32, lane, n_blk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? te1 : te0);
    }
    if (lane == 0) bulk_wait<0>();  // every staged store has completed
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Launches clusters of two CTAs, persistent: one pair per tile at most, and
// no more pairs than can be resident at once (queried once per device).
template <int EPI, int HD, bool F8>
cudaError_t launch_impl(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                        const CUtensorMap& tv, const GemmParams& p, int tiles, int sm_count,
                        cudaStream_t st) {
  static int max_pairs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<EPI>();
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_pairs[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<EPI, HD, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<EPI>());
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(2, 1, 1);
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<EPI, HD, F8>, &cfg) != cudaSuccess ||
        n <= 0) {
      (void)cudaGetLastError();
      n = sm_count / 2;
    }
    max_pairs[dev] = n < 1 ? 1 : n;
  }
  const int pairs = tiles < max_pairs[dev] ? tiles : max_pairs[dev];
  return launch_k(gemm_kernel<EPI, HD, F8>, dim3(2 * pairs, 1, 1), dim3(NUM_THREADS, 1, 1),
                  smem_bytes<EPI>(), st, 2, ta, tb, to, tv, p);
}

// Encodes the two operand maps (boxes of 128 bytes of K by 128 rows), counts
// the pair tiles and launches one persistent CTA pair per two SMs at most.
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
    const uint32_t box[2] = {BK, (uint32_t)BNH};
    if (!make_tmap(&tb, ES, B, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // the output map of the staged epilogues (unused by the others): fp32
  // boxes of 32 x 32 for the residual reduce-add, bf16 boxes of 64 x 32
  CUtensorMap to = ta;
  const bool resid = epi == EPI_RESIDUAL || epi == EPI_RESIDUAL_TANH || epi == EPI_RESIDUAL_SIGMOID;
  if (resid || glu || epi == EPI_BF16) {
    const uint32_t oes = resid ? 4 : 2;
    const uint64_t dims[2] = {(uint64_t)p.N, (uint64_t)p.M};
    const uint64_t strides[1] = {(uint64_t)p.ldo * oes};
    const uint32_t box[2] = {resid ? 32u : 64u, 32u};
    if (!make_tmap(&to, oes, p.out, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // EPI_QKV: q/k heads as [head][token][d] (boxes of 64 channels x 32 tokens
  // x 1 head, 128-byte swizzle like the staging buffers), and v transposed
  // [seq][g][c][s_pad] as a 2-D view x = token (s_len of s_pad columns),
  // y = (seq nkv + g) d + c (boxes of 32 tokens x d channels, unswizzled)
  CUtensorMap tv = ta;
  if (epi == EPI_QKV) {
    const QkvEpi& q = p.qkv;
    if (hd != 64 && hd != 128) return cudaErrorInvalidValue;
    {
      const uint64_t dims[3] = {(uint64_t)hd, (uint64_t)p.M, (uint64_t)(q.nh + q.nkv)};
      const uint64_t strides[2] = {(uint64_t)hd * 2, (uint64_t)p.M * hd * 2};
      const uint32_t box[3] = {64u, 32u, 1u};
      if (!make_tmap(&to, 2, q.qk, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
      const uint64_t n_seqs = (uint64_t)(p.M / q.s_len);
      const uint64_t dims[2] = {(uint64_t)q.s_len, n_seqs * q.nkv * hd};
      const uint64_t strides[1] = {(uint64_t)q.s_pad * 2};
      const uint32_t box[2] = {32u, (uint32_t)hd};
      if (!make_tmap(&tv, 2, q.vt, 2, dims, strides, box, false)) return cudaErrorInvalidValue;
    }
  }
  p.num_m = (p.M + PM - 1) / PM;
  p.num_n = glu ? p.N / 128 : (p.N + BN - 1) / BN;
  // raster groups of row blocks whose A rows take at most ~40 MB of L2
  {
    const long long a_bytes = (long long)PM * p.K * ES;
    long long g = (40ll << 20) / (a_bytes > 0 ? a_bytes : 1);
    if (g < 1) g = 1;
    p.group_m = g < p.num_m ? (int)g : p.num_m;
  }
  p.err = dev_err(ds);
  const int tiles = p.num_m * p.num_n;
  const int sms = ds->sm_count;
  switch (epi) {
    case EPI_BF16: return launch_impl<EPI_BF16, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_F32_BIAS: return launch_impl<EPI_F32_BIAS, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_RESIDUAL: return launch_impl<EPI_RESIDUAL, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_SWIGLU: return launch_impl<EPI_SWIGLU, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_GEGLU: return launch_impl<EPI_GEGLU, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_RESIDUAL_TANH: return launch_impl<EPI_RESIDUAL_TANH, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_RESIDUAL_SIGMOID:
      return launch_impl<EPI_RESIDUAL_SIGMOID, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
    case EPI_EULER:
      if constexpr (!F8) return launch_impl<EPI_EULER, 0, F8>(ta, tb, to, tv, p, tiles, sms, st);
      return cudaErrorInvalidValue;
    case EPI_QKV:
      if (hd == 64) return launch_impl<EPI_QKV, 64, F8>(ta, tb, to, tv, p, tiles, sms, st);
      if (hd == 128) return launch_impl<EPI_QKV, 128, F8>(ta, tb, to, tv, p, tiles, sms, st);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace dit
