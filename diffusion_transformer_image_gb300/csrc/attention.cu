// Non-causal flash attention on the fifth-generation tensor core.
//
// o_h = softmax(q_h k_g^T / sqrt(d)) v_g per sequence, no mask ([ERNIE]
// "Porting ERNIE-Image-Turbo to Zig and Metal", section VII, Decision 2),
// grouped KV heads g = h / (n_heads / n_kv_heads) ([ZFLOW] "From Python +
// CUDA to Pure Rust + Metal 4", section VI, attention(heads, kv_heads)).
//
// One CTA computes 128 query rows of one head of one sequence.  Roles:
//   warp 0      TMA producer of the q tile and of k tiles of 128 keys (a
//               two-stage ring released as soon as S_j = q k_j^T completes)
//   warp 6      TMA producer of v tiles (a two-stage ring released when
//               O += P_j v_j completes)
//   warp 1      TMEM allocator and MMA issuer: S_j = q k_j^T into one of two
//               TMEM score buffers, then O += P_j v_j into the TMEM output
//   warps 2..5  softmax: thread t owns query row t; reads S_j from TMEM,
//               keeps the running maximum and sum, writes P_j (bf16) to
//               shared memory in the swizzled layout the tensor core reads,
//               and rescales O in TMEM when the maximum grows by more than
//               2^8 (smaller growth is absorbed: exponentials stay <= 256)
// The issue order S_0, S_1, PV_0, S_2, PV_1, ... lets the softmax of block j
// overlap the tensor core work on blocks j + 1 and j - 1.
//
// v arrives transposed (vt[seq][g][c][key]) so that both MMAs read K-major
// operands.
#include <math_constants.h>

#include "internal.h"

namespace dit {
namespace {

constexpr int BQ = 128, BKV = 128;
constexpr int NUM_THREADS = 224;
constexpr float RESCALE_LOG2 = 8.0f;

template <int HD>
struct AttnLayout {
  static constexpr int Q_BYTES = BQ * HD * 2;     // HD/64 panels of 128 rows x 128 B
  static constexpr int K_BYTES = BKV * HD * 2;    // HD/64 panels of 128 keys x 128 B
  static constexpr int V_BYTES = HD * BKV * 2;    // 2 panels of HD rows x 64 keys
  static constexpr int V_PANEL = HD * 128;
  static constexpr int P_BYTES = BQ * BKV * 2;    // 2 panels of 128 rows x 64 keys
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + 2 * K_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * V_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int O_COL = 2 * BKV;           // TMEM columns: S0, S1, then O
};

struct AttnBars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t drain;
  uint32_t tmem_slot;
};

template <int HD>
constexpr size_t attn_smem_bytes() {
  return (size_t)AttnLayout<HD>::OFF_BAR + sizeof(AttnBars) + 1024 + 64;
}

struct AttnParams {
  __nv_bfloat16* o;
  int ldo;
  int s_len;
  int nh, nkv;
  float scale_log2;
  DevErr err;
};

template <int HD>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmV,
                const AttnParams p) {
  using L = AttnLayout<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  AttnBars* bars = reinterpret_cast<AttnBars*>(smem + L::OFF_BAR);

  const int warp = warp_id(), lane = lane_id();
  const int q0 = blockIdx.x * BQ;
  const int h = blockIdx.y;
  const int seq = blockIdx.z;
  const int g = h / (p.nh / p.nkv);
  const int nb = (p.s_len + BKV - 1) / BKV;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmQK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer: q, k
      mbar_arrive_expect_tx(&bars->q_full, L::Q_BYTES);
#pragma unroll
      for (int pn = 0; pn < HD / 64; ++pn)
        tma_load_3d(smem + L::OFF_Q + pn * 16384, &tmQK, &bars->q_full, h * HD + pn * 64, q0, seq);
      uint32_t filled = 0, fill_parity = 0;
      for (int j = 0; j < nb; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&bars->k_empty[st], ph ^ 1u, p.err)) break;
        uint8_t* sk = smem + L::OFF_K + st * L::K_BYTES;
        mbar_arrive_expect_tx(&bars->k_full[st], L::K_BYTES);
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn)
          tma_load_3d(sk + pn * 16384, &tmQK, &bars->k_full[st], (p.nh + g) * HD + pn * 64,
                      j * BKV, seq);
        filled |= 1u << st;
        fill_parity = (fill_parity & ~(1u << st)) | (ph << st);
      }
      // every copy issued must land before the CTA may exit
      mbar_wait(&bars->q_full, 0, p.err);
      for (int s = 0; s < 2; ++s)
        if (filled & (1u << s)) mbar_wait(&bars->k_full[s], (fill_parity >> s) & 1u, p.err);
    }
  } else if (warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------- TMA producer: v
      uint32_t filled = 0, fill_parity = 0;
      for (int j = 0; j < nb; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&bars->v_empty[st], ph ^ 1u, p.err)) break;
        uint8_t* sv = smem + L::OFF_V + st * L::V_BYTES;
        mbar_arrive_expect_tx(&bars->v_full[st], L::V_BYTES);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_3d(sv + pn * L::V_PANEL, &tmV, &bars->v_full[st], j * BKV + pn * 64, g * HD,
                      seq);
        filled |= 1u << st;
        fill_parity = (fill_parity & ~(1u << st)) | (ph << st);
      }
      for (int s = 0; s < 2; ++s)
        if (filled & (1u << s)) mbar_wait(&bars->v_full[s], (fill_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV);
      constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, HD);
      const uint32_t q_addr = smem_u32(smem + L::OFF_Q);
      const uint32_t o_tmem = tmem_base + L::O_COL;
      bool ok = mbar_wait(&bars->q_full, 0, p.err);
      for (int j = 0; j <= nb && ok; ++j) {
        if (j < nb) {
          const int st = j & 1;
          if (!mbar_wait(&bars->k_full[st], (j >> 1) & 1, p.err)) break;
          if (j >= 2 && !mbar_wait(&bars->s_free[st], ((j - 2) >> 1) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(smem + L::OFF_K + st * L::K_BYTES);
          const uint32_t s_tmem = tmem_base + st * BKV;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) {
            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
            umma_bf16(s_tmem, sdesc_sw128(q_addr + off), sdesc_sw128(k_addr + off), idesc_s, k > 0);
          }
          umma_commit(&bars->s_full[st]);
          umma_commit(&bars->k_empty[st]);
        }
        if (j >= 1) {
          const int i = j - 1;
          const int pb = i & 1;
          if (!mbar_wait(&bars->p_full[pb], (i >> 1) & 1, p.err)) break;
          if (!mbar_wait(&bars->v_full[pb], (i >> 1) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t p_addr = smem_u32(smem + L::OFF_P + pb * L::P_BYTES);
          const uint32_t v_addr = smem_u32(smem + L::OFF_V + pb * L::V_BYTES);
#pragma unroll
          for (int k = 0; k < BKV / 16; ++k) {
            const uint32_t poff = (k >> 2) * 16384 + (k & 3) * 32;
            const uint32_t voff = (k >> 2) * L::V_PANEL + (k & 3) * 32;
            umma_bf16(o_tmem, sdesc_sw128(p_addr + poff), sdesc_sw128(v_addr + voff), idesc_o,
                      (i > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars->pv_done[pb]);
          umma_commit(&bars->v_empty[pb]);
        }
      }
      umma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.err);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------------------------------------------- softmax warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row within the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_tmem = tmem_base + L::O_COL + lane_off;
    float m_used = -CUDART_INF_F;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&bars->s_full[sb], (j >> 1) & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BKV];
      __syncwarp();
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c)
        tmem_ld32(tmem_base + sb * BKV + lane_off + c * 32,
                  *reinterpret_cast<float(*)[32]>(&s[c * 32]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[sb]);

      const int kv0 = j * BKV;
      if (kv0 + BKV > p.s_len) {
#pragma unroll
        for (int c = 0; c < BKV; ++c)
          if (kv0 + c >= p.s_len) s[c] = -CUDART_INF_F;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < BKV; ++c) mx = fmaxf(mx, s[c]);
      mx *= p.scale_log2;

      const bool need = mx > m_used + RESCALE_LOG2;
      if (__any_sync(0xffffffffu, need) && j > 0) {
        // O holds PV_0 .. PV_{j-1}; wait for the last one, then rescale rows
        // whose maximum moved (alpha = 1 for the others).
        const float alpha = need ? ex2_approx(m_used - mx) : 1.0f;
        if (!mbar_wait(&bars->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float t[32];
          tmem_ld32(o_tmem + c * 32, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) t[i] *= alpha;
          tmem_st32(o_tmem + c * 32, t);
        }
        l *= alpha;
      }
      if (need) m_used = mx;

      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < BKV; ++c) {
        s[c] = ex2_approx(fmaf(s[c], p.scale_log2, -m_used));
        rs += s[c];
      }
      l += rs;

      // P buffer sb was last read by PV_{j-2}.
      if (j >= 2 && !mbar_wait(&bars->pv_done[sb], ((j - 2) >> 1) & 1, p.err)) {
        ok = false;
        break;
      }
      uint8_t* pbase = smem + L::OFF_P + sb * L::P_BYTES;
#pragma unroll
      for (int pn = 0; pn < 2; ++pn)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int k0 = pn * 64 + ch * 8;
          uint4 u;
          u.x = pack_bf16x2(s[k0 + 0], s[k0 + 1]);
          u.y = pack_bf16x2(s[k0 + 2], s[k0 + 3]);
          u.z = pack_bf16x2(s[k0 + 4], s[k0 + 5]);
          u.w = pack_bf16x2(s[k0 + 6], s[k0 + 7]);
          *reinterpret_cast<uint4*>(pbase + pn * 16384 + r * 128 + ((ch ^ (r & 7)) << 4)) = u;
        }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[sb]);
    }
    if (ok) {
      const int i = nb - 1;
      if (mbar_wait(&bars->pv_done[i & 1], (i >> 1) & 1, p.err)) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
        const int row = q0 + r;
        __nv_bfloat16* dst = p.o + ((size_t)seq * p.s_len + row) * p.ldo + h * HD;
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float t[32];
          tmem_ld32(o_tmem + c * 32, t);
          if (row < p.s_len) {
#pragma unroll
            for (int e = 0; e < 32; ++e) t[e] *= inv_l;
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 u;
              u.x = pack_bf16x2(t[8 * q + 0], t[8 * q + 1]);
              u.y = pack_bf16x2(t[8 * q + 2], t[8 * q + 3]);
              u.z = pack_bf16x2(t[8 * q + 4], t[8 * q + 5]);
              u.w = pack_bf16x2(t[8 * q + 6], t[8 * q + 7]);
              d4[q] = u;
            }
          }
          __syncwarp();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap& tq, const CUtensorMap& tv, const AttnParams& p,
                      dim3 grid, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)attn_smem_bytes<HD>());
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  attn_kernel<HD><<<grid, NUM_THREADS, attn_smem_bytes<HD>(), st>>>(tq, tv, p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(int hd, const __nv_bfloat16* qk, const __nv_bfloat16* vt,
                             int n_tokens, int n_seqs, int nh, int nkv, __nv_bfloat16* o,
                             cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  const int s_len = n_tokens / n_seqs;
  const int s_pad = (s_len + 7) & ~7;
  const uint64_t cqk = (uint64_t)(nh + nkv) * hd;
  CUtensorMap tq, tv;
  {
    const uint64_t dims[3] = {cqk, (uint64_t)s_len, (uint64_t)n_seqs};
    const uint64_t strides[2] = {cqk * 2, cqk * 2 * (uint64_t)s_len};
    const uint32_t box[3] = {64, BQ, 1};
    if (!make_tmap_bf16(&tq, qk, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)s_len, (uint64_t)nkv * hd, (uint64_t)n_seqs};
    const uint64_t strides[2] = {(uint64_t)s_pad * 2, (uint64_t)s_pad * 2 * nkv * hd};
    const uint32_t box[3] = {64, (uint32_t)hd, 1};
    if (!make_tmap_bf16(&tv, vt, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  AttnParams p;
  p.o = o;
  p.ldo = nh * hd;
  p.s_len = s_len;
  p.nh = nh;
  p.nkv = nkv;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)hd));
  p.err = dev_err(ds);
  dim3 grid((s_len + BQ - 1) / BQ, nh, n_seqs);
  if (hd == 64) return launch_hd<64>(tq, tv, p, grid, st);
  if (hd == 128) return launch_hd<128>(tq, tv, p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace dit
