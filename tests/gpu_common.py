"""Helpers shared by the GPU parity tests: device transfer, the parity
criteria, and oracle-side references built only from oracle functions."""
import numpy as np
import torch

from diffusion_transformer_image_gb300 import synth
from oracle import dit_oracle as O

F32 = np.float32


def dev():
    return torch.device("cuda:0")


def npf(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def pair_major_tables(ang):
    """Device cos/sin tables in the library's pair-major layout [d/2, n] from
    oracle angles [n, d/2]."""
    return (torch.from_numpy(np.ascontiguousarray(np.cos(ang).T)).to(dev()),
            torch.from_numpy(np.ascontiguousarray(np.sin(ang).T)).to(dev()))


def bf16_normal(shape, name, seed=7, std=1.0, mean=0.0) -> torch.Tensor:
    """Seeded bf16 CPU tensor (the oracle sees the same values widened)."""
    return synth.normal(shape, name, seed, std, mean).to(torch.bfloat16)


def max_err_vs_rms(got: np.ndarray, ref: np.ndarray):
    d = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    return float(d.max()), rms


def assert_block_parity(got, ref, frac=2e-2, what=""):
    """The per-block criterion: max|err| <= frac * RMS(reference output)."""
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err, rms = max_err_vs_rms(got, ref)
    assert err <= frac * rms, f"{what}: max|err| {err:.4e} > {frac} x RMS {rms:.4e}"
    return err / rms


def cosine(a, b):
    a = a.astype(np.float64).ravel()
    b = b.astype(np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def oracle_block_config(wl):
    return O.BlockConfig(wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.ffn,
                         rope_layout=wl.rope_layout, adaln=wl.adaln, qk_norm=wl.qk_norm,
                         norm_kind=wl.norm_kind, glu=wl.glu, rope_order=wl.rope_order,
                         gate_fn=wl.gate_fn, linear_format=wl.linear_format)


def oracle_weights(w: dict) -> dict:
    return {k: synth.to_numpy_f32(v) for k, v in w.items()}


def oracle_angles(wl):
    if wl.rope_layout == "half":
        return O.rope_angles_vit(wl.grid_h, wl.grid_w, wl.n_prefix, wl.head_dim)
    return O.rope_angles_3d(O.position_ids(wl.grid_h, wl.grid_w, wl.n_txt), wl.rope_axes,
                            wl.rope_theta)


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, F32)).to(torch.bfloat16).float().numpy()


def bf16_storage_rows(cfg, w, x, mod, angles, rows):
    """The block on sampled rows, evaluated with oracle functions in fp32 but
    with the intermediates the CUDA path stores in bf16 rounded to bf16: the
    GEMM inputs a and a2 (bf16 format only: the W8A8 format codes them from
    fp32), q/k/v, o and h.  Used only to size a tolerance: it measures how far
    bf16 storage alone moves the fp32 result (in the W8A8 format mostly
    through the e4m3 codes that it flips)."""
    shift1, scale1, gate1, shift2, scale2, gate2 = (mod[i] for i in range(6))
    gate1, gate2 = O.gate_act(gate1, cfg.gate_fn), O.gate_act(gate2, cfg.gate_fn)
    keep_a = cfg.linear_format == "w8a8_h256"
    rnd_a = (lambda t: t) if keep_a else _bf16
    a = rnd_a(O.modulate(O.norm(x, cfg.ln_eps, cfg.norm_kind), shift1, scale1))
    q, k, v = O.qkv_heads(cfg, a, w, angles)
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    o = _bf16(O.attention_rows(q[rows], k, v, cfg.n_heads, cfg.n_kv_heads))
    xr = O.gated_residual(x[rows], gate1, O.project(cfg, o, w["w_o"]))
    a2 = rnd_a(O.modulate(O.norm(xr, cfg.ln_eps, cfg.norm_kind), shift2, scale2))
    h = _bf16(O.glu(cfg, O.project(cfg, a2, w["w_gu"])))
    return O.gated_residual(xr, gate2, O.project(cfg, h, w["w_down"]))
