// Non-causal flash attention on the fifth-generation tensor core.
//
// o_h = softmax(q_h k_g^T / sqrt(d)) v_g per sequence, no mask ([ERNIE]
// "Porting ERNIE-Image-Turbo to Zig and Metal", section VII, Decision 2),
// grouped KV heads g = h / (n_heads / n_kv_heads) ([ZFLOW] "From Python +
// CUDA to Pure Rust + Metal 4", section VI, attention(heads, kv_heads)).
//
// One CTA computes two tiles of 128 query rows (A and B) of one head of one
// sequence, so every k/v tile loaded serves 256 queries: the kernel needs
// half the shared-memory ingress per FLOP of a one-tile design, which is
// what bounds a 128 x 128 attention block on this part.  Roles:
//   warp 0       TMA producer: both q tiles, then k tiles of 128 keys
//   warp 2       TMA producer: v tiles (transposed, 128 keys)
//   warp 1       TMEM allocator and MMA issuer, per key block j and tile t:
//                  O_t += P_t(j) v_j in two halves of 64 keys, each issued as
//                  soon as the softmax has stored that half of P (P read
//                  from TMEM), then
//                  S_t(j+1) = q_t k_{j+1}^T into the columns P_t(j) occupies
//                  (issue order is execution order on the tensor core).
//   warps 3..10  softmax, four per tile, one per TMEM lane quarter: thread r
//                owns query row r of its tile and all 128 scores of a block,
//                so the row maximum needs no exchange between threads.  It
//                keeps the running maximum and its row sum, overwrites S_t
//                with P_t (bf16, two per 32-bit column) one half at a time,
//                and rescales its row of O_t when the maximum grows by more
//                than 2^8 (smaller growth is absorbed: exponentials stay
//                <= 256).  While the softmax of one tile runs, the tensor
//                core works on the other tile.
// TMEM columns: S_A/P_A [0,128), S_B/P_B [128,256), O_A, O_B after them.
//
// q and k arrive head-major (qk[head][token][d], so a tile is one contiguous
// block) and v transposed (vt[seq][g][c][key]) so that both MMAs read K-major
// operands.
#include <math_constants.h>

#include "internal.h"

namespace dit {
namespace {

constexpr int BQ = 128, BKV = 128;
constexpr int NUM_SOFTMAX_WARPS = 8;    // 4 per query tile, one per TMEM lane quarter
constexpr int NUM_THREADS = (3 + NUM_SOFTMAX_WARPS) * 32;
constexpr float RESCALE_LOG2 = 8.0f;

// Ring depths per head width, sized to 227 KB of shared memory.
template <int HD>
struct AttnStages;
template <>
struct AttnStages<128> {
  static constexpr int K = 2, V = 2;
};
template <>
struct AttnStages<64> {
  static constexpr int K = 5, V = 5;
};

template <int HD>
struct AttnLayout {
  static constexpr int KS = AttnStages<HD>::K, VS = AttnStages<HD>::V;
  static constexpr int Q_BYTES = BQ * HD * 2;     // per tile: HD/64 panels of 128 rows x 128 B
  static constexpr int K_BYTES = BKV * HD * 2;    // HD/64 panels of 128 keys x 128 B
  static constexpr int V_BYTES = HD * BKV * 2;    // 2 panels of HD rows x 64 keys
  static constexpr int V_PANEL = HD * 128;
  static constexpr int OFF_Q = 0;                 // tile A, then tile B
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KS * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + VS * V_BYTES;
  static constexpr int END = OFF_BAR + 512;
  static constexpr int O_COL = 2 * BKV;           // O_A, then O_B
  static_assert(O_COL + 2 * HD <= 512, "TMEM overflow");
};

constexpr int MAX_STAGES = 6;

struct AttnBars {
  uint64_t q_full;
  uint64_t k_full[MAX_STAGES], k_empty[MAX_STAGES], v_full[MAX_STAGES], v_empty[MAX_STAGES];
  uint64_t s_full[2], pv_done[2];   // per query tile
  uint64_t p_half[2][2];            // per query tile and half of P (64 keys)
  uint64_t drain;
  uint32_t tmem_slot;
};

static_assert(sizeof(AttnBars) <= 512, "barrier block overflows its slot");

template <int HD>
constexpr size_t attn_smem_bytes() {
  return (size_t)AttnLayout<HD>::END + 1024;  // + slack to align the base to 1024 B
}

struct AttnParams {
  __nv_bfloat16* o;
  int ldo;
  int s_len, n_seqs;
  int nh, nkv;
  float scale_log2;
  DevErr err;
};

template <int HD>
__device__ __forceinline__ void issue_s(uint32_t s_tmem, uint32_t q_addr, uint32_t k_addr) {
  constexpr uint32_t idesc_s = idesc_bf16_f32(BQ, BKV);
#pragma unroll
  for (int k = 0; k < HD / 16; ++k) {
    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
    umma_bf16(s_tmem, sdesc_sw128(q_addr + off), sdesc_sw128(k_addr + off), idesc_s, k > 0);
  }
}

// O += P[:, 64 half : 64 half + 64] v[64 half : 64 half + 64, :]: four MMAs
// of 16 keys; P half h sits in TMEM columns [32 h, 32 h + 32), v's keys
// [64 h, 64 h + 64) in panel h of the stage.
template <int HD>
__device__ __forceinline__ void issue_pv_half(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_addr,
                                              int half, bool first) {
  using L = AttnLayout<HD>;
  constexpr uint32_t idesc_o = idesc_bf16_f32(BQ, HD);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const int k = half * 4 + kk;
    const uint32_t voff = (k >> 2) * L::V_PANEL + (k & 3) * 32;
    umma_bf16_ts(o_tmem, p_tmem + k * 8, sdesc_sw128(v_addr + voff), idesc_o,
                 (!first || k > 0) ? 1u : 0u);
  }
}

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
  const int q0 = blockIdx.x * 2 * BQ;
  const int h = blockIdx.y;
  const int seq = blockIdx.z;
  const int g = h / (p.nh / p.nkv);
  const int nb = (p.s_len + BKV - 1) / BKV;
  // Key blocks are visited starting at a block that depends on the query
  // tile, so the CTAs of one head stream different k/v tiles at any moment.
  // Softmax is order-independent; only the rounding order changes.
  const int kb0 = blockIdx.x % nb;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < MAX_STAGES; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->pv_done[t], 1);
      for (int hf = 0; hf < 2; ++hf) mbar_init(&bars->p_half[t][hf], NUM_SOFTMAX_WARPS / 2);
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
  grid_dep_wait();  // q, k and v of the projection before are complete
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer: q, k
      mbar_arrive_expect_tx(&bars->q_full, 2 * L::Q_BYTES);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn)
          tma_load_2d(smem + L::OFF_Q + t * L::Q_BYTES + pn * 16384, &tmQK, &bars->q_full,
                      pn * 64, (h * p.n_seqs + seq) * p.s_len + q0 + t * BQ);
      uint32_t filled = 0, fill_parity = 0;
      for (int j = 0; j < nb; ++j) {
        const int st = j % L::KS;
        const uint32_t ph = (j / L::KS) & 1;
        if (!mbar_wait(&bars->k_empty[st], ph ^ 1u, p.err)) break;
        uint8_t* sk = smem + L::OFF_K + st * L::K_BYTES;
        mbar_arrive_expect_tx(&bars->k_full[st], L::K_BYTES);
#pragma unroll
        for (int pn = 0; pn < HD / 64; ++pn)
          tma_load_2d(sk + pn * 16384, &tmQK, &bars->k_full[st], pn * 64,
                      ((p.nh + g) * p.n_seqs + seq) * p.s_len + ((j + kb0) % nb) * BKV);
        filled |= 1u << st;
        fill_parity = (fill_parity & ~(1u << st)) | (ph << st);
      }
      // every copy issued must land before the CTA may exit
      mbar_wait(&bars->q_full, 0, p.err);
      for (int s = 0; s < L::KS; ++s)
        if (filled & (1u << s)) mbar_wait(&bars->k_full[s], (fill_parity >> s) & 1u, p.err);
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------- TMA producer: v
      uint32_t filled = 0, fill_parity = 0;
      for (int j = 0; j < nb; ++j) {
        const int st = j % L::VS;
        const uint32_t ph = (j / L::VS) & 1;
        if (!mbar_wait(&bars->v_empty[st], ph ^ 1u, p.err)) break;
        uint8_t* sv = smem + L::OFF_V + st * L::V_BYTES;
        mbar_arrive_expect_tx(&bars->v_full[st], L::V_BYTES);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_2d(sv + pn * L::V_PANEL, &tmV, &bars->v_full[st],
                      ((j + kb0) % nb) * BKV + pn * 64, (seq * p.nkv + g) * HD);
        filled |= 1u << st;
        fill_parity = (fill_parity & ~(1u << st)) | (ph << st);
      }
      for (int s = 0; s < L::VS; ++s)
        if (filled & (1u << s)) mbar_wait(&bars->v_full[s], (fill_parity >> s) & 1u, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------- MMA issuer
      const uint32_t q_addr = smem_u32(smem + L::OFF_Q);
      bool ok = mbar_wait(&bars->q_full, 0, p.err) && mbar_wait(&bars->k_full[0], 0, p.err);
      if (ok) {
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + L::OFF_K);
        issue_s<HD>(tmem_base, q_addr, k_addr);
        umma_commit(&bars->s_full[0]);
        issue_s<HD>(tmem_base + BKV, q_addr + L::Q_BYTES, k_addr);
        umma_commit(&bars->s_full[1]);
        umma_commit(&bars->k_empty[0]);
      }
      // Per key block j, tile by tile: O_t += P_t(j) v_j half by half, then
      // S_t(j+1) (queued behind that PV).  Tile A's chain never waits on tile
      // B's softmax, so the two softmax groups alternate on the
      // special-function units while the tensor core works on the other tile.
      for (int j = 0; j < nb && ok; ++j) {
        const int vs = j % L::VS;
        const uint32_t v_addr = smem_u32(smem + L::OFF_V + vs * L::V_BYTES);
        const int st = (j + 1) % L::KS;
        const uint32_t k_addr = smem_u32(smem + L::OFF_K + st * L::K_BYTES);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t o_t = tmem_base + L::O_COL + t * HD;
          const uint32_t p_t = tmem_base + t * BKV;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (!mbar_wait(&bars->p_half[t][hf], j & 1, p.err) ||
                (t == 0 && hf == 0 && !mbar_wait(&bars->v_full[vs], (j / L::VS) & 1, p.err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv_half<HD>(o_t, p_t, v_addr, hf, j == 0);
          }
          if (!ok) break;
          umma_commit(&bars->pv_done[t]);
          if (t == 1) umma_commit(&bars->v_empty[vs]);
          if (j + 1 < nb) {
            // S_t(j+1) overwrites the columns P_t(j) occupies; the tensor core
            // performs one thread's MMAs in issue order, so PV_t(j) has read
            // P_t(j) before S_t(j+1) writes there and no wait is needed.
            if (t == 0 && !mbar_wait(&bars->k_full[st], ((j + 1) / L::KS) & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s<HD>(tmem_base + t * BKV, q_addr + t * L::Q_BYTES, k_addr);
            umma_commit(&bars->s_full[t]);
            if (t == 1) umma_commit(&bars->k_empty[st]);
          }
        }
      }
      umma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.err);
    }
  } else {
    // ---------------------------------------------------- softmax warps
    constexpr int OC = HD;       // output columns per thread (its whole row)
    const int t = (warp - 3) >> 2;       // query tile
    const int quarter = warp & 3;        // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;   // query row within the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem_base + t * BKV + lane_off;
    const uint32_t o_tmem = tmem_base + L::O_COL + t * HD + lane_off;
    float m_used = -CUDART_INF_F;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      if (!mbar_wait(&bars->s_full[t], j & 1, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BKV];
      __syncwarp();
      tmem_ld128(s_tmem, s);

      const int kv0 = ((j + kb0) % nb) * BKV;
      if (kv0 + BKV > p.s_len) {
#pragma unroll
        for (int c = 0; c < BKV; ++c)
          if (kv0 + c >= p.s_len) s[c] = -CUDART_INF_F;
      }
      // row maximum: chain i takes s[i], s[i + 16], ..., s[i + 112] with
      // three-input maxima
      float m16[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        m16[i] = fmax3(s[i], s[i + 16], s[i + 32]);
        m16[i] = fmax3(m16[i], s[i + 48], s[i + 64]);
        m16[i] = fmax3(m16[i], s[i + 80], s[i + 96]);
        m16[i] = fmaxf(m16[i], s[i + 112]);
      }
#pragma unroll
      for (int i = 0; i < 5; ++i) m16[i] = fmax3(m16[i], m16[i + 5], m16[i + 10]);
      const float mx =
          fmaxf(fmax3(m16[0], m16[1], m16[2]), fmax3(m16[3], m16[4], m16[15])) * p.scale_log2;

      const bool need = mx > m_used + RESCALE_LOG2;
      if (__any_sync(0xffffffffu, need) && j > 0) {
        // O_t holds PV up to block j - 1, complete: S_t(j) was issued after it.
        const float alpha = need ? ex2_approx(m_used - mx) : 1.0f;
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < OC / 16; ++c) {
          float tv[16];
          tmem_ld16(o_tmem + c * 16, tv);
#pragma unroll
          for (int i = 0; i < 16; ++i) tv[i] *= alpha;
          tmem_st16(o_tmem + c * 16, tv);
        }
        l *= alpha;
      }
      if (need) m_used = mx;

      // P_t(j) in bf16, two per 32-bit column, into the first half of S_t's
      // columns, 64 keys at a time: keys [64 h, 64 h + 64) land in columns
      // [32 h, 32 h + 32), and each half is handed to the MMA issuer as soon
      // as it is stored.  Exponent arguments and row sums two at a time
      // (packed fp32: each lane rounds exactly like the scalar fmaf / add).
      float2 r4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 nm2 = make_float2(-m_used, -m_used);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = hf * 64 + ch * 32;
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 x = __ffma2_rn(make_float2(s[c0 + c], s[c0 + c + 1]), sc2, nm2);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            r4[(c >> 1) & 3] = __fadd2_rn(r4[(c >> 1) & 3], e);
            pk[c / 2] = pack_bf16x2(e.x, e.y);
          }
          __syncwarp();
          tmem_st16u_nowait(s_tmem + c0 / 2, pk);
        }
        tmem_wait_st();   // this half of P is in TMEM before the MMA may read it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_half[t][hf]);
      }
      l += ((r4[0].x + r4[0].y) + (r4[1].x + r4[1].y)) + ((r4[2].x + r4[2].y) + (r4[3].x + r4[3].y));
    }
    if (ok) {
      if (mbar_wait(&bars->pv_done[t], (nb - 1) & 1, p.err)) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
        const int row = q0 + t * BQ + r;
        __nv_bfloat16* dst = p.o + ((size_t)seq * p.s_len + row) * p.ldo + h * HD;
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < OC / 32; ++c) {
          float tv[32];
          tmem_ld32(o_tmem + c * 32, tv);
          if (row < p.s_len) {
#pragma unroll
            for (int e = 0; e < 32; ++e) tv[e] *= inv_l;
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 u;
              u.x = pack_bf16x2(tv[8 * q + 0], tv[8 * q + 1]);
              u.y = pack_bf16x2(tv[8 * q + 2], tv[8 * q + 3]);
              u.z = pack_bf16x2(tv[8 * q + 4], tv[8 * q + 5]);
              u.w = pack_bf16x2(tv[8 * q + 6], tv[8 * q + 7]);
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
  return launch_k(attn_kernel<HD>, grid, dim3(NUM_THREADS), attn_smem_bytes<HD>(), st, 1, tq, tv, p);
}

}  // namespace

cudaError_t launch_attention(int hd, const __nv_bfloat16* qk, const __nv_bfloat16* vt,
                             int n_tokens, int n_seqs, int nh, int nkv, __nv_bfloat16* o,
                             cudaStream_t st) {
  const DeviceState* ds = device_state();
  if (!ds) return cudaErrorInitializationError;
  const int s_len = n_tokens / n_seqs;
  const int s_pad = (s_len + 7) & ~7;
  CUtensorMap tq, tv;
  {
    // q/k head-major [head][seq][token][d] as a 2D view: x = d, y = row of
    // (head * n_seqs + seq) * s_len + token.  A box that runs past the end
    // of a sequence reads the next sequence's rows: those keys are masked
    // and those query rows are never stored.
    const uint64_t dims[2] = {(uint64_t)hd, (uint64_t)(nh + nkv) * n_tokens};
    const uint64_t strides[1] = {(uint64_t)hd * 2};
    const uint32_t box[2] = {64, BQ};
    if (!make_tmap_bf16(&tq, qk, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    // v transposed [seq][g][c][s_pad] as a 2D view: x = key (only s_len of
    // the s_pad columns exist, the rest read as zero), y = (seq nkv + g) d + c
    const uint64_t dims[2] = {(uint64_t)s_len, (uint64_t)n_seqs * nkv * hd};
    const uint64_t strides[1] = {(uint64_t)s_pad * 2};
    const uint32_t box[2] = {64, (uint32_t)hd};
    if (!make_tmap_bf16(&tv, vt, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  AttnParams p;
  p.o = o;
  p.ldo = nh * hd;
  p.s_len = s_len;
  p.n_seqs = n_seqs;
  p.nh = nh;
  p.nkv = nkv;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)hd));
  p.err = dev_err(ds);
  dim3 grid((s_len + 2 * BQ - 1) / (2 * BQ), nh, n_seqs);
  if (hd == 64) return launch_hd<64>(tq, tv, p, grid, st);
  if (hd == 128) return launch_hd<128>(tq, tv, p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace dit
