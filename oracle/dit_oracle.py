"""CPU oracle for the diffusion-transformer hot path (test infrastructure only).

This module is the slow, obviously-correct definition that the CUDA path is
checked against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import it; the product library never does,
and it imports nothing from the product package.

Precision: float32 throughout, the precision the pages fix for their own
reference: the zml-flow-rs page's CPU f32 reference backend ("From Python +
CUDA to Pure Rust + Metal 4", §II and §X) runs the same graphs, and block
parity there is the bf16-vs-f32 gap.  Every
linear is one numpy float32 matmul (a library primitive); everything else is
written out step by step in the order the pages give it.  Inputs are the
seeded generator's bf16 values widened to float32; no intermediate is rounded.

Sources, cited by page title and section:
  [ERNIE]   "Porting ERNIE-Image-Turbo to Zig and Metal: An 8B Diffusion
            Transformer From Scratch on Apple Silicon"
  [ZFLOW]   "From Python + CUDA to Pure Rust + Metal 4: How zml-flow-rs Stops
            Us Writing a Kernel Per Model"
  [MAKEPAD] makepad commit log for libs/ai/metal/shaders/ggml (resident
            pre-norm ViT backbone commit)

Readings taken where the pages are silent or disagree:
  * every norm is LayerNorm without affine (eps 1e-6); per-head qk-LayerNorm
    has a gain and bias over head_dim;
  * qk-LayerNorm is applied before RoPE ([ZFLOW] §VI: the fused per-head norm
    kernel normalises each head, then rotates it);
  * RoPE pairs are interleaved inside each axis chunk for the DiT, and
    rotate-half (pairs i, i+d/2) for the ViT;
  * the FFN is SwiGLU: silu(gate) * up, gate rows first in the stacked weight;
  * gates are applied as plain products (identity gate function);
  * one modulation vector [6, H] is shared by all layers of a step;
  * image rows come first in the joint sequence, then text rows;
  * the W8A8 format with H256 rotation ([ZFLOW] §VII) rotates the
    contraction axis of both operands in independent 256-wide blocks by the
    orthonormal Sylvester Hadamard matrix and codes each row with one scale
    (amax / 448); the 8-bit code is e4m3, the 8-bit type the target tensor
    cores multiply (they have no integer kind).

Parity pins: every function here is checked by tests/test_oracle_pins.py
against closed forms, brute force or invariants.  The numeric value of a
whole block or a whole 36-layer step has no printed worked example on the
pages: "parity unpinned" for those composites beyond the invariants that the
pin tests check.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np

F32 = np.float32


def _map(fn: Callable, items: Sequence) -> list:
    """[fn(i) for i in items] on a thread pool over the host's cores.  Used
    only for pieces of work that are independent by definition (one attention
    head of one sequence; one chunk of rows of a row-wise coding): each piece
    computes exactly what the serial loop computes, numpy releases the
    interpreter lock inside its kernels, and the pool exists only for the
    duration of the call."""
    items = list(items)
    n = min(len(items), os.cpu_count() or 1)
    if n <= 1:
        return [fn(i) for i in items]
    with ThreadPoolExecutor(n) as ex:
        return list(ex.map(fn, items))


def _row_chunks(n_rows: int) -> list:
    """Row ranges that split n_rows into about four pieces per host core."""
    parts = max(1, min(n_rows, 4 * (os.cpu_count() or 1)))
    step = -(-n_rows // parts)
    return [(r, min(r + step, n_rows)) for r in range(0, n_rows, step)]


# --------------------------------------------------------------------------
# Configuration (shapes and semantics of one block / one model)
# --------------------------------------------------------------------------
@dataclass
class BlockConfig:
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    rope_layout: str = "interleaved"   # "interleaved" (DiT) or "half" (ViT)
    adaln: bool = True                  # 6-way AdaLN modulation + gates
    qk_norm: bool = True                # per-head norm on q and k
    ln_eps: float = 1e-6
    # Variants of the block as the ERNIE page draws it ([ERNIE] §IV per-layer
    # graph, §V Bug 1) and of the gates the zml-flow-rs page discovers
    # ([ZFLOW] §IV, §V).  The defaults are the workload's block.
    norm_kind: str = "layer"            # "layer" or "rms": pre-norms, qk-norm, final norm
    glu: str = "silu"                   # "silu" or "gelu_tanh" (clamped tanh GELU)
    rope_order: str = "norm_rope"       # "norm_rope" or "rope_norm"
    gate_fn: str = "identity"           # "identity", "tanh" or "sigmoid"
    # Format of the four projections ([ZFLOW] §VII): "bf16", or "w8a8_h256":
    # both operands rotated by a 256-point Hadamard along K and coded in 8 bits
    # with one scale per row.
    linear_format: str = "bf16"


@dataclass
class ModelConfig:
    block: BlockConfig
    n_layers: int
    latent_channels: int = 128
    t_dim: int = 256
    t_scale: float = 1000.0
    rope_axes: Sequence[int] = field(default_factory=lambda: (32, 48, 48))
    rope_theta: float = 256.0


# --------------------------------------------------------------------------
# Elementary steps
# --------------------------------------------------------------------------
def linear(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None) -> np.ndarray:
    """y = x W^T (+ b) with W stored [out, in]; the dense linear of
    [ZFLOW] §VI (Backend::linear).  One float32 matmul."""
    y = np.matmul(x.astype(F32, copy=False), w.astype(F32, copy=False).T)
    if b is not None:
        y = y + b.astype(F32, copy=False)
    return y.astype(F32, copy=False)


# --------------------------------------------------------------------------
# Low-precision linears: Hadamard rotation and 8-bit codes ([ZFLOW] §VII)
# --------------------------------------------------------------------------
HADAMARD_N = 256
E4M3_MAX = 448.0


def fwht256_rows(x: np.ndarray) -> np.ndarray:
    """x H along the last axis, in independent blocks of 256, where H is the
    256-point Sylvester Hadamard matrix scaled by 1/16 (so H H^T = I): the
    rotation "H256" of [ZFLOW] §VII.  Computed by the fast Walsh-Hadamard
    transform in float32: eight butterfly stages, span 1, 2, ..., 128, each
    replacing the pair (u at index i, w at index i + span), i without the span
    bit, by (u + w, u - w); then one exact multiplication by 1/16."""
    y = np.array(x, dtype=F32, copy=True)
    n, k = y.shape
    if k % HADAMARD_N:
        raise ValueError("the rotated axis must be a multiple of 256")
    nb = k // HADAMARD_N
    span = 1
    while span < HADAMARD_N:
        t = y.reshape(n, nb, HADAMARD_N // (2 * span), 2, span)
        u = t[:, :, :, 0, :].copy()
        w = t[:, :, :, 1, :].copy()
        t[:, :, :, 0, :] = u + w
        t[:, :, :, 1, :] = u - w
        span *= 2
    return (y * F32(1.0 / 16.0)).astype(F32)


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Rounds float32 values to the nearest value of the 8-bit float format
    e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinity,
    largest finite 448, subnormals in steps of 2^-9), ties to the even
    mantissa, magnitudes above 448 saturated to 448.  Returns float32 values
    on that grid (each is one code)."""
    a = np.abs(v.astype(np.float64))
    _, e = np.frexp(a)                       # a = m 2^e, m in [0.5, 1)
    e = np.maximum(e - 1, -6)                # binade exponent; subnormals share -6
    step = np.ldexp(1.0, e - 3)              # 3 mantissa bits
    q = np.rint(a / step) * step             # rint: half to even; a / step is exact
    q = np.minimum(q, E4M3_MAX)
    return (np.sign(v) * q).astype(F32)


def e4m3_decode_table() -> np.ndarray:
    """The value of each of the 256 e4m3 codes as float32 (code = sign << 7 |
    exponent << 3 | mantissa); the two NaN codes 0x7f and 0xff map to NaN."""
    vals = np.empty(256, dtype=F32)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        if e == 15 and m == 7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = s * m * 2.0 ** -9
        else:
            vals[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def quantize_rows_e4m3(y: np.ndarray):
    """Per-row 8-bit coding ([ZFLOW] §VII: "per-row" on both operands).
    For each row: amax = max |y|; scale = amax / 448 and inv = 448 / amax, both
    one float32 division; code = e4m3_round(y * inv) with the product in
    float32.  An all-zero row gets scale 0 and zero codes.  Returns (the codes'
    values as float32 [rows, k], scale float32 [rows]); y ~= code * scale."""
    y = y.astype(F32, copy=False)
    amax = np.max(np.abs(y), axis=1).astype(F32)
    nz = amax > 0
    safe = np.where(nz, amax, F32(1.0)).astype(F32)
    scale = np.where(nz, (safe / F32(E4M3_MAX)).astype(F32), F32(0.0)).astype(F32)
    inv = np.where(nz, (F32(E4M3_MAX) / safe).astype(F32), F32(0.0)).astype(F32)
    codes = e4m3_round((y * inv[:, None]).astype(F32))
    return codes, scale


def rotate_quantize(x: np.ndarray):
    """Rotation then per-row coding of one operand: quantize_rows_e4m3 of
    fwht256_rows(x).  Both steps work on each row alone, so chunks of rows
    are coded independently and stacked."""
    x = x.astype(F32, copy=False)
    parts = _map(lambda r: quantize_rows_e4m3(fwht256_rows(x[r[0]:r[1]])), _row_chunks(x.shape[0]))
    return (np.concatenate([p[0] for p in parts], axis=0),
            np.concatenate([p[1] for p in parts], axis=0))


def linear_w8a8_h256(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T in the format W8A8 with H256 rotation ([ZFLOW] §VII): by the
    rotation rule (x H)(W H)^T = x W^T for orthogonal H, both operands are
    rotated along K and coded per row; y[i, o] = sx[i] sw[o] sum_k qx[i, k]
    qw[o, k].  The sum of code products is taken in float64, where it is
    exact for these operand sizes."""
    qx, sx = rotate_quantize(x)
    qw, sw = rotate_quantize(w)
    acc = np.matmul(qx.astype(np.float64), qw.astype(np.float64).T)
    return (acc * sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]).astype(F32)


def project(cfg: "BlockConfig", x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """One of the block's four projections in the block's linear format."""
    if cfg.linear_format == "bf16":
        return linear(x, w)
    if cfg.linear_format == "w8a8_h256":
        return linear_w8a8_h256(x, w)
    raise ValueError(cfg.linear_format)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x / (1 + e^-x), the activation of the SwiGLU FFN
    ([ZFLOW] §VI, Oak's SwiGLU GEMM) and of the time-embedding MLP."""
    x = x.astype(F32, copy=False)
    with np.errstate(over="ignore"):
        return (x / (F32(1.0) + np.exp(-x))).astype(F32)


def layer_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis without affine:
    (v - mean) / sqrt(var + eps), biased variance.  The pre-norm of the
    AdaLN-Zero block ([ERNIE] §IV per-layer graph); LayerNorm is the norm the
    workload specifies."""
    x = x.astype(F32, copy=False)
    mean = x.mean(axis=-1, keepdims=True, dtype=F32)
    d = x - mean
    var = (d * d).mean(axis=-1, keepdims=True, dtype=F32)
    return (d / np.sqrt(var + F32(eps))).astype(F32)


def rms_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis without affine: v / sqrt(mean(v^2) + eps)
    (the norm the ERNIE page draws for AdaLN-Zero and qk-norm, [ERNIE] §IV)."""
    x = x.astype(F32, copy=False)
    ms = (x * x).mean(axis=-1, keepdims=True, dtype=F32)
    return (x / np.sqrt(ms + F32(eps))).astype(F32)


def norm(x: np.ndarray, eps: float, kind: str) -> np.ndarray:
    """The block's norm: LayerNorm or RMSNorm (BlockConfig.norm_kind)."""
    if kind == "layer":
        return layer_norm(x, eps)
    if kind == "rms":
        return rms_norm(x, eps)
    raise ValueError(kind)


def gelu_tanh_clamped(x: np.ndarray) -> np.ndarray:
    """GELU by its tanh approximation with the two clamps of [ERNIE] §V Bug 1:
    a = sqrt(2/pi) (x + 0.044715 x^3) limited to [-20, 20] (tanh is already
    saturated there, and the limit keeps half-precision tanh finite), then
    0.5 x (1 + tanh a) limited to the half-precision range [-65504, 65504]."""
    x = x.astype(F32, copy=False)
    k = F32(0.7978845608)
    a = np.clip(k * (x + F32(0.044715) * x * x * x), F32(-20.0), F32(20.0)).astype(F32)
    y = F32(0.5) * x * (F32(1.0) + np.tanh(a))
    return np.clip(y, F32(-65504.0), F32(65504.0)).astype(F32)


def gate_act(g: np.ndarray, fn: str) -> np.ndarray:
    """The gate function applied to a modulation gate before it scales its
    branch: identity (ERNIE, [ERNIE] §VII Decision 1), tanh (Qwen-Image,
    [ZFLOW] §IV) or sigmoid (Krea-2, [ZFLOW] §V)."""
    g = g.astype(F32, copy=False)
    if fn == "identity":
        return g
    if fn == "tanh":
        return np.tanh(g).astype(F32)
    if fn == "sigmoid":
        with np.errstate(over="ignore"):
            return (F32(1.0) / (F32(1.0) + np.exp(-g))).astype(F32)
    raise ValueError(fn)


def modulate(xn: np.ndarray, shift: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """AdaLN modulation xn * (1 + scale) + shift ([ERNIE] §V Bug 4: the
    `norm(x) * (1 + scale) + shift` form; [ZFLOW] §VI `plus_one`)."""
    return (xn * (F32(1.0) + scale.astype(F32)) + shift.astype(F32)).astype(F32)


def gated_residual(x: np.ndarray, gate: Optional[np.ndarray], y: np.ndarray) -> np.ndarray:
    """x + gate * y in float32 ([ERNIE] §VII Decision 1, f32 residual stream).
    gate None means a plain residual (pre-norm ViT, [MAKEPAD])."""
    if gate is None:
        return (x + y).astype(F32)
    return (x + gate.astype(F32) * y).astype(F32)


# --------------------------------------------------------------------------
# Positions and rotary embedding
# --------------------------------------------------------------------------
def position_ids(grid_h: int, grid_w: int, n_txt: int, image_first: bool = True) -> np.ndarray:
    """Per-token 3-axis positions ([ERNIE] §IV Token Layout and §VII
    Decision 3): an image token at grid cell (h, w) gets (n_txt, h, w); text
    token j gets (j, 0, 0).  Image rows come first in the joint sequence.
    Returns int32 [grid_h*grid_w + n_txt, 3]."""
    img = np.zeros((grid_h * grid_w, 3), dtype=np.int32)
    for i in range(grid_h * grid_w):
        img[i, 0] = n_txt
        img[i, 1] = i // grid_w
        img[i, 2] = i % grid_w
    txt = np.zeros((n_txt, 3), dtype=np.int32)
    for j in range(n_txt):
        txt[j, 0] = j
    return np.concatenate([img, txt] if image_first else [txt, img], axis=0)


def rope_angles_3d(pos: np.ndarray, axes: Sequence[int], theta: float) -> np.ndarray:
    """Rotation angle of every pair for multi-axis RoPE ([ERNIE] §I: 3D RoPE
    with axes [32,48,48], theta=256).  The head vector is split into
    consecutive chunks of sizes axes[0], axes[1], axes[2]; pair j of axis a
    turns by pos[a] * theta^(-2j / axes[a]).  Angles in float32 ([ZFLOW] §V:
    RoPE tables are built in F32).  Returns float32 [N, sum(axes)/2]."""
    n = pos.shape[0]
    cols = []
    for a, d_a in enumerate(axes):
        j = np.arange(d_a // 2, dtype=np.float64)
        inv_freq = (theta ** (-2.0 * j / d_a)).astype(F32)          # [d_a/2]
        p = pos[:, a].astype(F32)[:, None]                          # [N,1]
        cols.append((p * inv_freq[None, :]).astype(F32))
    out = np.concatenate(cols, axis=1)
    assert out.shape == (n, sum(axes) // 2)
    return out


def rope_angles_vit(grid_h: int, grid_w: int, n_prefix: int, head_dim: int,
                    base: float = 10000.0) -> np.ndarray:
    """Angle table for the pre-norm ViT's rotate-half RoPE, which [MAKEPAD]
    applies from precomputed tables.  The pages give no formula; the reading
    taken: prefix (cls/register) tokens are unrotated (angle 0); patch token
    (r, c) uses pairs k < d/4 with angle r * w_k and pairs d/4 <= k < d/2 with
    angle c * w_(k-d/4), w_k = base^(-k/(d/4)).  Returns float32
    [n_prefix + grid_h*grid_w, d/2]."""
    q = head_dim // 4
    k = np.arange(q, dtype=np.float64)
    w = (base ** (-k / q)).astype(F32)
    n = n_prefix + grid_h * grid_w
    ang = np.zeros((n, head_dim // 2), dtype=F32)
    for t in range(grid_h * grid_w):
        r, c = t // grid_w, t % grid_w
        ang[n_prefix + t, :q] = F32(r) * w
        ang[n_prefix + t, q:] = F32(c) * w
    return ang


def rope_apply(x: np.ndarray, angles: np.ndarray, layout: str) -> np.ndarray:
    """Rotate pairs of x [..., N, d] by angles [N, d/2].
    interleaved: pair k is (x[2k], x[2k+1]); half: pair k is (x[k], x[k+d/2]).
    Each pair (a, b) -> (a cos - b sin, a sin + b cos)."""
    c = np.cos(angles).astype(F32)
    s = np.sin(angles).astype(F32)
    d = x.shape[-1]
    out = np.empty_like(x, dtype=F32)
    if layout == "interleaved":
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
    elif layout == "half":
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c - b * s
        out[..., d // 2:] = a * s + b * c
    else:
        raise ValueError(layout)
    return out


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int,
              n_kv_heads: int, n_seqs: int = 1) -> np.ndarray:
    """Non-causal joint attention with no mask ([ERNIE] §VII Decision 2) and
    grouped KV heads ([ZFLOW] §VI Backend::attention(heads, kv_heads)).

    q: [N, n_heads, d]; k, v: [N, n_kv_heads, d]; N = n_seqs * S, tokens of
    sequence s are rows [s*S, (s+1)*S) and attend only within their sequence
    (one image per sequence for the batched ViT).  Query head h reads KV head
    h // (n_heads / n_kv_heads).  Exact two-pass softmax of q.k / sqrt(d) in
    float32.  Returns [N, n_heads * d]."""
    n, _, d = q.shape
    s_len = n // n_seqs
    group = n_heads // n_kv_heads
    scale = F32(1.0 / math.sqrt(d))
    out = np.empty((n, n_heads, d), dtype=F32)

    def one_head(sh):  # sequence s, query head h (independent of the others)
        s, h = sh
        rows = slice(s * s_len, (s + 1) * s_len)
        g = h // group
        sc = np.matmul(q[rows, h, :], k[rows, g, :].T).astype(F32) * scale
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc).astype(F32)
        p = p / p.sum(axis=1, keepdims=True, dtype=F32)
        out[rows, h, :] = np.matmul(p, v[rows, g, :])

    _map(one_head, [(s, h) for s in range(n_seqs) for h in range(n_heads)])
    return out.reshape(n, n_heads * d)


def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int,
                   n_kv_heads: int) -> np.ndarray:
    """The same attention for a subset of query rows of one sequence:
    q_rows [R, n_heads, d] attend to all keys k, v [S, n_kv_heads, d].  Each
    output row depends only on its own query, so this equals the matching
    rows of attention() (pinned by a test).  Returns [R, n_heads * d]."""
    r, _, d = q_rows.shape
    group = n_heads // n_kv_heads
    scale = F32(1.0 / math.sqrt(d))
    out = np.empty((r, n_heads, d), dtype=F32)

    def one_head(h):
        g = h // group
        sc = np.matmul(q_rows[:, h, :], k[:, g, :].T).astype(F32) * scale
        sc = sc - sc.max(axis=1, keepdims=True)
        p = np.exp(sc).astype(F32)
        p = p / p.sum(axis=1, keepdims=True, dtype=F32)
        out[:, h, :] = np.matmul(p, v[:, g, :])

    _map(one_head, range(n_heads))
    return out.reshape(r, n_heads * d)


# --------------------------------------------------------------------------
# One block
# --------------------------------------------------------------------------
def qkv_heads(cfg: BlockConfig, a: np.ndarray, w: dict, angles: np.ndarray):
    """QKV projection, per-head qk-norm (gain, bias over head_dim) and RoPE
    on q and k ([ERNIE] §IV per-layer graph).  Order norm-then-RoPE by
    default ([ZFLOW] §VI, the fused per-head norm then rotation); the ERNIE
    page draws RoPE then qk-norm (rope_order "rope_norm").  Returns
    q [N,nh,d], k, v [N,nkv,d]."""
    nh, nkv, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    n = a.shape[0]
    qkv = project(cfg, a, w["w_qkv"])
    q = qkv[:, : nh * d].reshape(n, nh, d)
    k = qkv[:, nh * d: (nh + nkv) * d].reshape(n, nkv, d)
    v = qkv[:, (nh + nkv) * d:].reshape(n, nkv, d)
    def qk_norm(t, g, b):
        return norm(t, cfg.ln_eps, cfg.norm_kind) * g + b

    def rotate(t):  # angles are per token; broadcast over heads
        return np.ascontiguousarray(np.swapaxes(
            rope_apply(np.swapaxes(t, 0, 1), angles, cfg.rope_layout), 0, 1))

    if cfg.rope_order == "norm_rope":
        if cfg.qk_norm:
            q = qk_norm(q, w["q_g"], w["q_b"])
            k = qk_norm(k, w["k_g"], w["k_b"])
        q, k = rotate(q), rotate(k)
    elif cfg.rope_order == "rope_norm":
        q, k = rotate(q), rotate(k)
        if cfg.qk_norm:
            q = qk_norm(q, w["q_g"], w["q_b"])
            k = qk_norm(k, w["k_g"], w["k_b"])
    else:
        raise ValueError(cfg.rope_order)
    return q.astype(F32), k.astype(F32), v.astype(F32)


def block_forward(cfg: BlockConfig, w: dict, x: np.ndarray,
                  mod: Optional[np.ndarray], angles: np.ndarray,
                  n_seqs: int = 1) -> np.ndarray:
    """One transformer block, steps in the order of [ERNIE] §IV:
    AdaLN -> QKV -> qk-norm -> RoPE -> attention -> out-projection -> gated
    residual -> AdaLN -> gate/up -> GLU -> down -> gated residual.

    x: float32 [N, H] residual stream (returned updated, input untouched).
    mod: [6, H] = [shift1, scale1, gate1, shift2, scale2, gate2] ([ERNIE]
    §IV: the adaLN split), or None for the pre-norm ViT, whose norms carry a
    gain and bias (ln1_g, ln1_b, ln2_g, ln2_b) and whose residuals are plain.
    angles: [N, d/2] RoPE angles per token (per token within the sequence
    when n_seqs > 1: shape [S, d/2])."""
    x = x.astype(F32, copy=True)
    n = x.shape[0]
    if angles.shape[0] != n:
        angles = np.tile(angles, (n // angles.shape[0], 1))
    if cfg.adaln:
        shift1, scale1, gate1, shift2, scale2, gate2 = (mod[i] for i in range(6))
        gate1, gate2 = gate_act(gate1, cfg.gate_fn), gate_act(gate2, cfg.gate_fn)
        a = modulate(norm(x, cfg.ln_eps, cfg.norm_kind), shift1, scale1)
    else:
        gate1 = gate2 = None
        a = norm(x, cfg.ln_eps, cfg.norm_kind) * w["ln1_g"] + w["ln1_b"]
    q, k, v = qkv_heads(cfg, a, w, angles)
    o = attention(q, k, v, cfg.n_heads, cfg.n_kv_heads, n_seqs)
    x = gated_residual(x, gate1, project(cfg, o, w["w_o"]))
    if cfg.adaln:
        a = modulate(norm(x, cfg.ln_eps, cfg.norm_kind), shift2, scale2)
    else:
        a = norm(x, cfg.ln_eps, cfg.norm_kind) * w["ln2_g"] + w["ln2_b"]
    x = gated_residual(x, gate2, project(cfg, glu(cfg, project(cfg, a, w["w_gu"])), w["w_down"]))
    return x


def glu(cfg: BlockConfig, gu: np.ndarray) -> np.ndarray:
    """The gated FFN activation on the stacked gate/up projection (gate
    columns first): SiLU(gate) * up ([ZFLOW] §VI, SwiGLU) or the clamped
    tanh GELU(gate) * up ([ERNIE] §IV and §V Bug 1)."""
    f = cfg.ffn
    act = silu if cfg.glu == "silu" else gelu_tanh_clamped
    if cfg.glu not in ("silu", "gelu_tanh"):
        raise ValueError(cfg.glu)
    return (act(gu[:, :f]) * gu[:, f:]).astype(F32)


def block_forward_rows(cfg: BlockConfig, w: dict, x: np.ndarray, mod: Optional[np.ndarray],
                       angles: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """block_forward restricted to some output rows of a single sequence:
    keys and values come from every row, everything after attention is
    per-row.  Same steps and order as block_forward; returns [len(rows), H]
    (pinned against block_forward by a test)."""
    x = x.astype(F32, copy=False)
    if cfg.adaln:
        shift1, scale1, gate1, shift2, scale2, gate2 = (mod[i] for i in range(6))
        gate1, gate2 = gate_act(gate1, cfg.gate_fn), gate_act(gate2, cfg.gate_fn)
        a = modulate(norm(x, cfg.ln_eps, cfg.norm_kind), shift1, scale1)
    else:
        gate1 = gate2 = None
        a = norm(x, cfg.ln_eps, cfg.norm_kind) * w["ln1_g"] + w["ln1_b"]
    q, k, v = qkv_heads(cfg, a, w, angles)
    o = attention_rows(q[rows], k, v, cfg.n_heads, cfg.n_kv_heads)
    xr = gated_residual(x[rows], gate1, project(cfg, o, w["w_o"]))
    if cfg.adaln:
        a2 = modulate(norm(xr, cfg.ln_eps, cfg.norm_kind), shift2, scale2)
    else:
        a2 = norm(xr, cfg.ln_eps, cfg.norm_kind) * w["ln2_g"] + w["ln2_b"]
    return gated_residual(xr, gate2,
                          project(cfg, glu(cfg, project(cfg, a2, w["w_gu"])), w["w_down"]))


# --------------------------------------------------------------------------
# Timestep conditioning
# --------------------------------------------------------------------------
def timestep_embedding(t: float, dim: int = 256, max_period: float = 10000.0) -> np.ndarray:
    """Sinusoidal timestep embedding with flip_sin_to_cos ([ZFLOW] §IV: the
    timestep sinusoid is `flip_sin_to_cos`): [cos(t w_j), sin(t w_j)] with
    w_j = max_period^(-j/half), j < half = dim/2, cosine half first."""
    half = dim // 2
    j = np.arange(half, dtype=np.float64)
    w = np.exp(-math.log(max_period) * j / half).astype(F32)
    arg = (F32(t) * w).astype(F32)
    return np.concatenate([np.cos(arg), np.sin(arg)]).astype(F32)


def conditioning(mw: dict, sigma: float, t_dim: int, t_scale: float):
    """Timestep MLP and the two modulation heads, once per step:
    temb = W2 SiLU(W1 e + b1) + b2 with e the sinusoid of T = t_scale*sigma;
    mod = Wm SiLU(temb) + bm reshaped [6, H] (shared by every layer);
    final = Wf SiLU(temb) + bf reshaped [2, H] = [scale, shift]
    ([ERNIE] §IV adaLN split; §V Bug 4 final-norm chunk order)."""
    e = timestep_embedding(F32(t_scale) * F32(sigma), t_dim)
    temb = linear(silu(linear(e[None, :], mw["t_w1"], mw["t_b1"])), mw["t_w2"], mw["t_b2"])
    st = silu(temb)
    mod = linear(st, mw["mod_w"], mw["mod_b"]).reshape(6, -1)
    fin = linear(st, mw["fin_w"], mw["fin_b"]).reshape(2, -1)
    return mod, fin


# --------------------------------------------------------------------------
# Flow-matching scheduler
# --------------------------------------------------------------------------
def flowmatch_sigmas(n_steps: int, shift: float) -> np.ndarray:
    """Shifted flow-matching sigmas ([ERNIE] §I: FlowMatchEulerDiscrete with
    shift=4.0, exponential time shift).  s_i = 1 - i/n_steps, i = 0..n_steps;
    the exponential shift with mu = ln(shift) maps s to
    e^mu / (e^mu + 1/s - 1) = shift*s / (1 + (shift-1)*s), and s = 0 to 0.
    Computed in float64, returned float32 [n_steps + 1]."""
    out = np.zeros(n_steps + 1, dtype=np.float64)
    for i in range(n_steps + 1):
        s = 1.0 - i / n_steps
        out[i] = shift * s / (1.0 + (shift - 1.0) * s)
    return out.astype(F32)


def euler_step(x: np.ndarray, v: np.ndarray, sigma: float, sigma_next: float) -> np.ndarray:
    """Flow-matching Euler update x + (sigma_next - sigma) * v, sign +1
    ([ZFLOW] §IV Euler sign +1, §V `euler = primitive`).  Float32, the
    product rounded before the add."""
    dt = F32(F32(sigma_next) - F32(sigma))
    return (x.astype(F32) + (dt * v.astype(F32)).astype(F32)).astype(F32)


# --------------------------------------------------------------------------
# Whole denoise step (DiT) and ViT forward
# --------------------------------------------------------------------------
def final_layer(x_img: np.ndarray, fin: np.ndarray, w_out: np.ndarray,
                b_out: np.ndarray, eps: float, kind: str = "layer") -> np.ndarray:
    """AdaLN-continuous final norm and output projection: chunk order
    [scale, shift] ([ERNIE] §V Bug 4), then the linear back to the latent
    channels.  The norm kind follows the blocks'."""
    scale, shift = fin[0], fin[1]
    return linear(modulate(norm(x_img, eps, kind), shift, scale), w_out, b_out)


def denoise_step(mc: ModelConfig, mw: dict, latent: np.ndarray, text: np.ndarray,
                 grid_h: int, grid_w: int, sigma: float, sigma_next: float,
                 n_layers: Optional[int] = None, return_velocity: bool = False):
    """One flow-matching Euler step of the DiT ([ERNIE] §IV: latent
    [4096,128] -> 36 layers -> velocity; 8 such steps).

    latent: float32 [grid_h*grid_w, C]; text: float32 [n_txt, H].
    mw: model weights dict with 'patch_w' [H,C], 'patch_b', 't_w1', 't_b1',
    't_w2', 't_b2', 'mod_w', 'mod_b', 'fin_w', 'fin_b', 'out_w' [C,H], 'out_b'
    and 'layers' (a sequence of per-block dicts, read one at a time).
    Returns the new latent (and the velocity if asked)."""
    bc = mc.block
    n_img = grid_h * grid_w
    n_txt = text.shape[0]
    mod, fin = conditioning(mw, sigma, mc.t_dim, mc.t_scale)
    x_img = linear(latent, mw["patch_w"], mw["patch_b"])
    x = np.concatenate([x_img, text.astype(F32)], axis=0)
    angles = rope_angles_3d(position_ids(grid_h, grid_w, n_txt), mc.rope_axes, mc.rope_theta)
    layers = mw["layers"]
    nl = mc.n_layers if n_layers is None else n_layers
    for li in range(nl):
        x = block_forward(bc, layers[li], x, mod, angles)
    v = final_layer(x[:n_img], fin, mw["out_w"], mw["out_b"], bc.ln_eps, bc.norm_kind)
    new = euler_step(latent, v, sigma, sigma_next)
    return (new, v) if return_velocity else new


def vit_forward(bc: BlockConfig, layers: Sequence[dict], x: np.ndarray,
                angles: np.ndarray, n_seqs: int, n_layers: Optional[int] = None) -> np.ndarray:
    """Pre-norm ViT stack ([MAKEPAD]: LayerNorm, q/k/v, rotate-half RoPE from
    tables, attention, out, LayerNorm, SwiGLU, down; residuals in place).
    x: [n_seqs * S, H]; attention stays within each image's S tokens."""
    nl = len(layers) if n_layers is None else n_layers
    for li in range(nl):
        x = block_forward(bc, layers[li], x, None, angles, n_seqs)
    return x
