"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and names workload shapes; it holds
none of the method's arithmetic (no norms, rotary angles, positions,
modulation or attention).  Every tensor gets its own sub-seed derived from
(name, seed), so one tensor never depends on the order others were drawn in.

Distributions follow the workload definitions: linears N(0, 0.02) stored as
bf16 (round-to-nearest-even), activations N(0, 1), norm gains 1 + N(0, 0.02)
and norm biases N(0, 0.02) (a gain drawn from N(0, 0.02) would zero q and k
and make attention degenerate).
"""
from __future__ import annotations

import os
import zlib
from dataclasses import dataclass, field
from typing import Dict, List, Sequence

import torch


@dataclass(frozen=True)
class Workload:
    """Shapes of one synthetic workload."""
    name: str
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    rope_axes: Sequence[int] = (32, 48, 48)
    rope_theta: float = 256.0
    rope_layout: str = "interleaved"
    adaln: bool = True
    qk_norm: bool = True
    grid_h: int = 64
    grid_w: int = 64
    n_txt: int = 256
    n_layers: int = 1
    n_steps: int = 0
    shift: float = 4.0
    latent_channels: int = 128
    t_dim: int = 256
    n_seqs: int = 1          # images per batch (ViT); the DiT uses one sequence
    n_prefix: int = 0        # ViT cls/register tokens per image
    t_block: float = 0.5     # timestep of the single-block workloads
    norm_kind: str = "layer"  # block variants (see the oracle's BlockConfig)
    glu: str = "silu"
    rope_order: str = "norm_rope"
    gate_fn: str = "identity"
    linear_format: str = "bf16"  # or "w8a8_h256" (the projections' 8-bit format)

    @property
    def seq_len(self) -> int:
        return self.n_prefix + self.grid_h * self.grid_w + self.n_txt

    @property
    def n_tokens(self) -> int:
        return self.n_seqs * self.seq_len

    @property
    def qkv_width(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


WORKLOADS: Dict[str, Workload] = {
    # one block, 16x16 image grid, no text, hidden 256, 4x64 heads, FFN 768
    "tiny_block": Workload("tiny_block", 256, 4, 4, 64, 768, rope_axes=(16, 24, 24),
                           grid_h=16, grid_w=16, n_txt=0),
    # ERNIE-shaped block: 4096 image + 256 text tokens, hidden 4096, 32x128, FFN 12288
    "ernie_block": Workload("ernie_block", 4096, 32, 32, 128, 12288),
    # ERNIE-shaped 8B DiT: 36 blocks, 8 Euler steps, shift 4
    "ernie_full": Workload("ernie_full", 4096, 32, 32, 128, 12288, n_layers=36, n_steps=8),
    # Krea-2-shaped GQA DiT at 512^2: 32x32 grid + 256 text, hidden 6144, 48q/8kv heads
    "krea_gqa": Workload("krea_gqa", 6144, 48, 8, 128, 16384, grid_h=32, grid_w=32,
                         n_layers=28, n_steps=8),
    # pre-norm ViT: 4 images x (5 prefix + 32x32 patches), hidden 1024, 16x64, FFN 4096
    "vit_backbone": Workload("vit_backbone", 1024, 16, 16, 64, 4096, rope_axes=(),
                             rope_layout="half", adaln=False, qk_norm=False,
                             grid_h=32, grid_w=32, n_txt=0, n_layers=24,
                             n_seqs=4, n_prefix=5),
}


def sub_seed(name: str, seed: int) -> int:
    return zlib.crc32(f"{name}:{seed}".encode()) & 0x7FFFFFFF


def normal(shape, name: str, seed: int, std: float = 1.0, mean: float = 0.0,
           device="cpu") -> torch.Tensor:
    """float32 N(mean, std^2) tensor from its own seeded generator."""
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(name, seed))
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def bf16_valued(t: torch.Tensor) -> torch.Tensor:
    """float32 tensor whose values are exactly bf16-representable."""
    return t.to(torch.bfloat16).to(torch.float32)


def block_weights(wl: Workload, layer: int, seed: int = 0, device="cpu",
                  std: float = 0.02) -> Dict[str, torch.Tensor]:
    """One block's weights: bf16 linears [out, in]; float32 norm params."""
    p = f"L{layer}."
    d, h, f = wl.head_dim, wl.hidden, wl.ffn
    w = {
        "w_qkv": bf16(normal((wl.qkv_width, h), p + "w_qkv", seed, std, device=device)),
        "w_o": bf16(normal((h, wl.n_heads * d), p + "w_o", seed, std, device=device)),
        "w_gu": bf16(normal((2 * f, h), p + "w_gu", seed, std, device=device)),
        "w_down": bf16(normal((h, f), p + "w_down", seed, std, device=device)),
    }
    if wl.qk_norm:
        for n in ("q", "k"):
            w[n + "_g"] = bf16_valued(normal((d,), p + n + "_g", seed, std, 1.0, device=device))
            w[n + "_b"] = bf16_valued(normal((d,), p + n + "_b", seed, std, device=device))
    if not wl.adaln:
        for n in ("ln1", "ln2"):
            w[n + "_g"] = bf16_valued(normal((h,), p + n + "_g", seed, std, 1.0, device=device))
            w[n + "_b"] = bf16_valued(normal((h,), p + n + "_b", seed, std, device=device))
    return w


def model_weights(wl: Workload, seed: int = 0, device="cpu", std: float = 0.02,
                  mod_bias_std: float = 0.02, n_layers: int = None) -> Dict[str, object]:
    """Head/tail weights of the DiT (patch embed, time MLP, modulation heads,
    output projection; biases float32) and the per-layer block weights."""
    h, c, td = wl.hidden, wl.latent_channels, wl.t_dim
    nl = wl.n_layers if n_layers is None else n_layers
    w: Dict[str, object] = {
        "patch_w": bf16(normal((h, c), "patch_w", seed, std, device=device)),
        "patch_b": bf16_valued(normal((h,), "patch_b", seed, std, device=device)),
        "t_w1": bf16(normal((h, td), "t_w1", seed, std, device=device)),
        "t_b1": bf16_valued(normal((h,), "t_b1", seed, std, device=device)),
        "t_w2": bf16(normal((h, h), "t_w2", seed, std, device=device)),
        "t_b2": bf16_valued(normal((h,), "t_b2", seed, std, device=device)),
        "mod_w": bf16(normal((6 * h, h), "mod_w", seed, std, device=device)),
        "mod_b": bf16_valued(normal((6 * h,), "mod_b", seed, mod_bias_std, device=device)),
        "fin_w": bf16(normal((2 * h, h), "fin_w", seed, std, device=device)),
        "fin_b": bf16_valued(normal((2 * h,), "fin_b", seed, mod_bias_std, device=device)),
        "out_w": bf16(normal((c, h), "out_w", seed, std, device=device)),
        "out_b": bf16_valued(normal((c,), "out_b", seed, std, device=device)),
    }
    w["layers"] = _layers(wl, nl, seed, device, std)
    return w


def _layers(wl: Workload, n_layers: int, seed: int, device, std: float) -> List[Dict]:
    """Every layer's weights.  On the host the layers are drawn on a thread
    pool (each tensor has its own generator, so the values do not depend on
    the order or the thread they are drawn in)."""
    if torch.device(device).type != "cpu" or n_layers <= 1:
        return [block_weights(wl, li, seed, device, std) for li in range(n_layers)]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(min(n_layers, os.cpu_count() or 1)) as ex:
        return list(ex.map(lambda li: block_weights(wl, li, seed, device, std), range(n_layers)))


def residual_input(wl: Workload, seed: int = 1, device="cpu") -> torch.Tensor:
    """x ~ N(0,1), float32 with bf16-representable values, [n_tokens, H]."""
    return bf16_valued(normal((wl.n_tokens, wl.hidden), "x", seed, device=device))


def modulation_input(wl: Workload, seed: int = 1, std: float = 0.5,
                     device="cpu") -> torch.Tensor:
    """A direct [6, H] modulation input for single-block runs (float32)."""
    return bf16_valued(normal((6, wl.hidden), "mod", seed, std, device=device))


def text_input(wl: Workload, seed: int = 1, device="cpu") -> torch.Tensor:
    """Synthetic text sequence [n_txt, H] ~ N(0,1), bf16."""
    return bf16(normal((wl.n_txt, wl.hidden), "text", seed, device=device))


def latent_input(wl: Workload, seed: int = 1, device="cpu") -> torch.Tensor:
    """Initial latent noise [grid_h*grid_w, C] ~ N(0,1), float32."""
    return normal((wl.grid_h * wl.grid_w, wl.latent_channels), "latent", seed, device=device)


def to_numpy_f32(t: torch.Tensor):
    return t.detach().to("cpu", torch.float32).numpy()
