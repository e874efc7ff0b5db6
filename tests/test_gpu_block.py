"""Block and denoise-step parity on the GPU against the oracle.

Per-block criterion: max|err| <= 2e-2 x RMS(oracle output).  Small cases are
compared element by element on every output; the full-size workloads are
compared on sampled rows that the oracle computes one by one (keys and
values from every row, everything after attention per row)."""
import dataclasses

import numpy as np
import pytest
import torch

from diffusion_transformer_image_gb300 import synth
from gpu_common import (assert_block_parity, bf16_storage_rows, cosine, dev, max_err_vs_rms, npf,
                        oracle_angles, oracle_block_config, oracle_weights)
from oracle import dit_oracle as O

pytestmark = pytest.mark.gpu

dit = pytest.importorskip("diffusion_transformer_image_gb300.dit")


def small(name, **kw):
    return synth.Workload(name, **kw)


SMALL_BLOCKS = {
    "tiny_block": synth.WORKLOADS["tiny_block"],
    "gqa_small": small("gqa_small", hidden=512, n_heads=4, n_kv_heads=2, head_dim=128, ffn=1024,
                       grid_h=12, grid_w=12, n_txt=16),
    "vit_small": small("vit_small", hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=512,
                       rope_axes=(), rope_layout="half", adaln=False, qk_norm=False, grid_h=8,
                       grid_w=8, n_txt=0, n_seqs=2, n_prefix=5),
}


def rope_tables(wl):
    half = wl.head_dim // 2
    c = torch.empty(half, wl.seq_len, device=dev())
    s = torch.empty(half, wl.seq_len, device=dev())
    if wl.rope_layout == "half":
        dit.dit_rope_table_vit(wl.grid_h, wl.grid_w, wl.n_prefix, wl.head_dim, 10000.0, c, s)
    else:
        dit.dit_rope_table_grid(wl.grid_h, wl.grid_w, wl.n_txt, wl.rope_axes, wl.rope_theta, c, s)
    return c, s


def run_block_gpu(wl, w, x, mod):
    """mod: device tensor [6, H], a CPU tensor, or None (pre-norm ViT)."""
    cfg = dit.block_config_from(wl)
    blk = dit.DeviceBlock(w, dev(), wl.linear_format)
    rc, rs = rope_tables(wl)
    xg = x.to(dev()).contiguous()
    dit.dit_block_forward(cfg, blk, xg, None if mod is None else mod.to(dev()).contiguous(), rc,
                          rs, n_seqs=wl.n_seqs)
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    return npf(xg)


def conditioning_pair(wl, sigma):
    """The block's modulation from the seeded timestep MLP at `sigma`,
    computed independently by each side: the GPU conditioning kernels and the
    oracle's conditioning().  Returns (device [6, H], oracle [6, H])."""
    mw = synth.model_weights(wl, seed=0, n_layers=0)
    cfg = dit.model_config_from(wl, 0)
    model = dit.DeviceModel(mw, dev(), layers=[])
    H = wl.hidden
    mod = torch.empty(6, H, device=dev())
    fin = torch.empty(2, H, device=dev())
    scratch = torch.empty(wl.t_dim + 2 * H, device=dev())
    dit.dit_timestep_conditioning(cfg, model, sigma, mod, fin, scratch)
    ow = {k: synth.to_numpy_f32(v) for k, v in mw.items() if k != "layers"}
    rmod, _ = O.conditioning(ow, sigma, wl.t_dim, 1000.0)
    return mod, rmod


@pytest.mark.parametrize("name", list(SMALL_BLOCKS))
def test_block_forward_small(name):
    """Every output of a small block; AdaLN blocks take their modulation from
    the timestep MLP at t = 0.5 (T = 500)."""
    wl = SMALL_BLOCKS[name]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = conditioning_pair(wl, wl.t_block) if wl.adaln else (None, None)
    got = run_block_gpu(wl, w, x, mod_g)
    ref = O.block_forward(oracle_block_config(wl), oracle_weights(w), npf(x), mod_o,
                          oracle_angles(wl), wl.n_seqs)
    assert_block_parity(got, ref, what=name)


@pytest.mark.parametrize("name", ["tiny_block", "gqa_small"])
def test_block_forward_small_strong_modulation(name):
    """Every output, with a direct N(0, 0.5^2) modulation so that the gates
    and (1 + scale) are large and every branch weighs on the output."""
    wl = SMALL_BLOCKS[name]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod = synth.modulation_input(wl, seed=1)
    got = run_block_gpu(wl, w, x, mod)
    ref = O.block_forward(oracle_block_config(wl), oracle_weights(w), npf(x), npf(mod),
                          oracle_angles(wl), wl.n_seqs)
    assert_block_parity(got, ref, what=name)


VARIANTS = {
    # the block as the ERNIE page draws it: RMSNorm, RoPE then qk-norm,
    # clamped tanh-GELU GLU
    "ernie_as_drawn": dict(norm_kind="rms", rope_order="rope_norm", glu="gelu_tanh"),
    "tanh_gate": dict(gate_fn="tanh"),
    "sigmoid_gate": dict(gate_fn="sigmoid"),
}


def with_variant(wl, **kw):
    import dataclasses
    return dataclasses.replace(wl, **kw)


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("name", ["tiny_block", "gqa_small"])
def test_block_variants_small(name, variant):
    wl = with_variant(SMALL_BLOCKS[name], **VARIANTS[variant])
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = conditioning_pair(wl, wl.t_block)
    got = run_block_gpu(wl, w, x, mod_g)
    ref = O.block_forward(oracle_block_config(wl), oracle_weights(w), npf(x), mod_o,
                          oracle_angles(wl), wl.n_seqs)
    assert_block_parity(got, ref, what=f"{name}/{variant}")


def test_ernie_as_drawn_block_full_size():
    """The ERNIE-shaped block as the page draws it, at full size, 74 valid text
    tokens (4096 + 74 = 4170 rows: ragged GEMM and attention tails) as when the
    text is truncated to its valid length ([ERNIE] section VII, Decision 2);
    every row against the oracle's block (assert_full_size_parity)."""
    wl = with_variant(synth.WORKLOADS["ernie_block"], n_txt=74, **VARIANTS["ernie_as_drawn"])
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = conditioning_pair(wl, wl.t_block)
    got = run_block_gpu(wl, w, x, mod_g)
    assert_full_size_parity(wl, w, x, got, mod_o, "ernie_as_drawn 4170")


def test_block_truncated_text_4170_rows():
    """The workload's block with the text truncated to 74 tokens: 4170 rows,
    every row against the oracle's block (assert_full_size_parity)."""
    wl = with_variant(synth.WORKLOADS["ernie_block"], n_txt=74)
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = conditioning_pair(wl, wl.t_block)
    got = run_block_gpu(wl, w, x, mod_g)
    assert_full_size_parity(wl, w, x, got, mod_o, "4170 rows")


def test_block_zero_gates_pass_through_exactly():
    wl = synth.WORKLOADS["tiny_block"]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod = synth.modulation_input(wl, seed=1)
    mod[2] = 0.0
    mod[5] = 0.0
    got = run_block_gpu(wl, w, x, mod)
    np.testing.assert_array_equal(got, npf(x))


def test_block_token_permutation_equivariance():
    # Non-causal attention with position-only RoPE: permuting rows together
    # with their positions permutes the output.
    wl = synth.WORKLOADS["tiny_block"]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod = synth.modulation_input(wl, seed=1).to(dev())
    cfg = dit.block_config_from(wl)
    blk = dit.DeviceBlock(w, dev())
    pos = torch.from_numpy(O.position_ids(wl.grid_h, wl.grid_w, wl.n_txt))
    perm = torch.randperm(wl.n_tokens, generator=torch.Generator().manual_seed(3))
    outs = []
    for p in (torch.arange(wl.n_tokens), perm):
        c = torch.empty(wl.head_dim // 2, wl.n_tokens, device=dev())
        s = torch.empty_like(c)
        dit.dit_rope_table_pos(pos[p].contiguous().to(dev()), wl.rope_axes, wl.rope_theta, c, s)
        xg = x[p].contiguous().to(dev())
        dit.dit_block_forward(cfg, blk, xg, mod, c, s)
        outs.append(npf(xg))
    assert_block_parity(outs[1], outs[0][perm.numpy()], frac=1e-2, what="permutation")


def test_block_position_offset_invariance():
    # RoPE encodes relative positions: shifting every token's position by one
    # vector leaves a non-causal block's output unchanged (up to bf16
    # rounding flips of q and k, far inside the bound below).
    wl = synth.WORKLOADS["tiny_block"]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod = synth.modulation_input(wl, seed=1).to(dev())
    cfg = dit.block_config_from(wl)
    blk = dit.DeviceBlock(w, dev())
    pos = torch.from_numpy(O.position_ids(wl.grid_h, wl.grid_w, wl.n_txt))
    deltas = []
    for off in ((0, 0, 0), (5, 3, 11)):
        p = (pos + torch.tensor(off, dtype=torch.int32)).contiguous().to(dev())
        c = torch.empty(wl.head_dim // 2, wl.n_tokens, device=dev())
        s = torch.empty_like(c)
        dit.dit_rope_table_pos(p, wl.rope_axes, wl.rope_theta, c, s)
        xg = x.to(dev()).contiguous()
        dit.dit_block_forward(cfg, blk, xg, mod, c, s)
        deltas.append(npf(xg) - npf(x))
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    assert_block_parity(deltas[1], deltas[0], frac=2e-2, what="position offset")


def test_gqa_equals_mha_with_repeated_kv_heads():
    # Query head h reads kv head h // (n_heads / n_kv_heads): repeating each
    # kv head's k and v projection rows for its group of query heads gives a
    # block with n_kv_heads = n_heads that computes the same thing.
    gqa = synth.Workload("gqa_rep", 256, 8, 2, 64, 512, rope_axes=(16, 24, 24), grid_h=8,
                         grid_w=8, n_txt=8)
    mha = dataclasses.replace(gqa, name="mha_rep", n_kv_heads=8)
    nh, nkv, d = 8, 2, 64
    w = synth.block_weights(gqa, 0, seed=0)
    q, k, v = w["w_qkv"].split([nh * d, nkv * d, nkv * d])

    def rep(t):
        return t.reshape(nkv, d, -1).repeat_interleave(nh // nkv, dim=0).reshape(nh * d, -1)

    w_mha = dict(w)
    w_mha["w_qkv"] = torch.cat([q, rep(k), rep(v)]).contiguous()
    x = synth.residual_input(gqa, seed=1)
    mod = synth.modulation_input(gqa, seed=1)
    got_gqa = run_block_gpu(gqa, w, x, mod) - npf(x)
    got_mha = run_block_gpu(mha, w_mha, x, mod) - npf(x)
    assert_block_parity(got_gqa, got_mha, frac=1e-3, what="GQA vs repeated MHA")


def test_block_equals_its_stages():
    # dit_block_forward enqueues the same kernels as its stage entry points:
    # norm, QKV with qk-norm and RoPE, attention, gated out projection, norm,
    # SwiGLU, gated down projection.  Same inputs, same order: bit-identical.
    wl = SMALL_BLOCKS["gqa_small"]
    n, H, F, d = wl.n_tokens, wl.hidden, wl.ffn, wl.head_dim
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod = synth.modulation_input(wl, seed=1).to(dev()).contiguous()
    cfg = dit.block_config_from(wl)
    blk = dit.DeviceBlock(w, dev())
    rc, rs = rope_tables(wl)
    xb = x.to(dev()).contiguous()
    dit.dit_block_forward(cfg, blk, xb, mod, rc, rs)
    xs = x.to(dev()).contiguous()
    a = torch.empty(n, H, dtype=torch.bfloat16, device=dev())
    qk = torch.empty(wl.n_heads + wl.n_kv_heads, n, d, dtype=torch.bfloat16, device=dev())
    vt = torch.empty(1, wl.n_kv_heads, d, (n + 7) // 8 * 8, dtype=torch.bfloat16, device=dev())
    o = torch.empty(n, wl.n_heads * d, dtype=torch.bfloat16, device=dev())
    h = torch.empty(n, F, dtype=torch.bfloat16, device=dev())
    dit.dit_ln_modulate(0, xs, mod[0], mod[1], 1e-6, a)
    dit.dit_qkv_rope(cfg, blk, a, rc, rs, qk, vt)
    dit.dit_attention(cfg, qk, vt, o)
    dit.dit_linear(dit.DIT_EPI_RESIDUAL, o, blk.t["w_o"], xs, mod[2])
    dit.dit_ln_modulate(0, xs, mod[3], mod[4], 1e-6, a)
    dit.dit_linear(dit.DIT_EPI_SWIGLU, a, blk.t["w_gu"], h)
    dit.dit_linear(dit.DIT_EPI_RESIDUAL, h, blk.t["w_down"], xs, mod[5])
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    np.testing.assert_array_equal(npf(xs), npf(xb))


def assert_full_size_parity(wl, w, x, got, mod_o, what):
    """Every row of a full-size block against the oracle: max|err| within the
    stated per-block bound, 2e-2 x RMS, or, where bf16 storage of the GEMM
    inputs alone moves the worst element further than that, within 1.25 x
    the error of an fp32 evaluation that rounds the same intermediates to
    bf16 (built from oracle functions only)."""
    cfg, ow, ang = oracle_block_config(wl), oracle_weights(w), oracle_angles(wl)
    ref = O.block_forward(cfg, ow, npf(x), mod_o, ang, wl.n_seqs)
    sim = bf16_storage_rows(cfg, ow, npf(x), mod_o, ang, np.arange(wl.n_tokens))
    e_gpu, rms = max_err_vs_rms(got, ref)
    e_sim, _ = max_err_vs_rms(sim, ref)
    print(f"{what}: every row, max|err| {e_gpu / rms:.4f} x RMS, bf16 storage alone "
          f"{e_sim / rms:.4f} x RMS")
    assert e_gpu <= max(2e-2 * rms, 1.25 * e_sim + 1e-3 * rms), (e_gpu / rms, e_sim / rms)


def sample_rows(n):
    rng = np.random.default_rng(11)
    return np.unique(np.concatenate([[0, 127, 128, n - 257, n - 256, n - 1],
                                     rng.choice(n, 42, replace=False)]))


@pytest.mark.parametrize("name", ["ernie_block", "krea_gqa"])
def test_block_forward_full_size(name):
    """The 4352-token ERNIE-shaped block and the 1280-token Krea-shaped GQA
    block at full size, in the launch configuration the bench uses, with the
    modulation of the timestep MLP at t = 0.5; every row against the oracle's
    block (assert_full_size_parity)."""
    wl = synth.WORKLOADS[name]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = conditioning_pair(wl, wl.t_block)
    got = run_block_gpu(wl, w, x, mod_g)
    assert_full_size_parity(wl, w, x, got, mod_o, name)


@pytest.mark.parametrize("name", ["ernie_block", "krea_gqa"])
def test_block_forward_full_size_strong_modulation(name):
    """Full size with a direct N(0, 0.5^2) modulation.  Here the bf16 storage
    of the GEMM inputs (a, q/k/v, o, h) alone moves the fp32 result by about
    2.5-3 % of RMS, so the bound is derived from that arithmetic: the error
    may not exceed 1.25 x the error of an fp32 evaluation that rounds the same
    intermediates to bf16 (computed from oracle functions only)."""
    wl = synth.WORKLOADS[name]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod = synth.modulation_input(wl, seed=1)
    got = run_block_gpu(wl, w, x, mod)
    rows = sample_rows(wl.n_tokens)
    cfg, ow, ang = oracle_block_config(wl), oracle_weights(w), oracle_angles(wl)
    ref = O.block_forward_rows(cfg, ow, npf(x), npf(mod), ang, rows)
    sim = bf16_storage_rows(cfg, ow, npf(x), npf(mod), ang, rows)
    e_gpu, rms = max_err_vs_rms(got[rows], ref)
    e_sim, _ = max_err_vs_rms(sim, ref)
    assert e_gpu <= 1.25 * e_sim + 1e-3 * rms, (e_gpu / rms, e_sim / rms)


def test_vit_block_full_size():
    """The pre-norm ViT block at full size: 4 images x (5 + 32x32) tokens."""
    wl = synth.WORKLOADS["vit_backbone"]
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    got = run_block_gpu(wl, w, x, None)
    ref = O.block_forward(oracle_block_config(wl), oracle_weights(w), npf(x), None,
                          oracle_angles(wl), wl.n_seqs)
    assert_block_parity(got, ref, what="vit_backbone")


# ------------------------------------------------------------ denoise step
def oracle_model_config(wl, n_layers):
    return O.ModelConfig(block=oracle_block_config(wl), n_layers=n_layers,
                         latent_channels=wl.latent_channels, t_dim=wl.t_dim,
                         rope_axes=wl.rope_axes, rope_theta=wl.rope_theta)


class _LazyLayers:
    """Per-layer oracle weights converted on access, so a 36-layer model never
    sits in host memory as fp32 all at once."""

    def __init__(self, layers):
        self.layers = layers

    def __len__(self):
        return len(self.layers)

    def __getitem__(self, i):
        return oracle_weights(self.layers[i])


def oracle_model_weights(mw):
    out = {k: synth.to_numpy_f32(v) for k, v in mw.items() if k != "layers"}
    out["layers"] = _LazyLayers(mw["layers"])
    return out


def run_denoise(wl, n_layers, sigma, sigma_next):
    mw = synth.model_weights(wl, seed=0, n_layers=n_layers)
    latent = synth.latent_input(wl, seed=1)
    text = synth.text_input(wl, seed=1)
    cfg = dit.model_config_from(wl, n_layers)
    model = dit.DeviceModel(mw, dev(), linear_format=wl.linear_format)
    lat = latent.to(dev()).contiguous()
    v = torch.empty_like(lat)
    dit.dit_denoise_step(cfg, model, lat, text.to(dev()) if wl.n_txt else None, wl.grid_h,
                         wl.grid_w, sigma, sigma_next, velocity_out=v)
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    new_ref, v_ref = O.denoise_step(oracle_model_config(wl, n_layers), oracle_model_weights(mw),
                                    npf(latent), npf(text), wl.grid_h, wl.grid_w, sigma,
                                    sigma_next, return_velocity=True)
    return npf(lat), npf(v), new_ref, v_ref, npf(latent)


TINY_DIT = small("tiny_dit", hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=768,
                 rope_axes=(16, 24, 24), grid_h=8, grid_w=8, n_txt=16, n_layers=2,
                 latent_channels=32)


def test_timestep_conditioning():
    wl = TINY_DIT
    mw = synth.model_weights(wl, seed=0, n_layers=0)
    cfg = dit.model_config_from(wl, 0)
    model = dit.DeviceModel(mw, dev(), layers=[])
    H = wl.hidden
    mod = torch.empty(6 * H, device=dev())
    fin = torch.empty(2 * H, device=dev())
    scratch = torch.empty(wl.t_dim + 2 * H, device=dev())
    s = float(O.flowmatch_sigmas(8, 4.0)[3])
    dit.dit_timestep_conditioning(cfg, model, s, mod, fin, scratch)
    rmod, rfin = O.conditioning(oracle_model_weights(dict(mw, layers=[])), s, wl.t_dim, 1000.0)
    np.testing.assert_allclose(npf(mod), rmod.ravel(), rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(npf(fin), rfin.ravel(), rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("step", [0, 5])
def test_denoise_step_tiny(step):
    s = O.flowmatch_sigmas(8, 4.0)
    lat, v, new_ref, v_ref, lat0 = run_denoise(TINY_DIT, 2, float(s[step]), float(s[step + 1]))
    assert_block_parity(v, v_ref, what="velocity")
    # latent update: parity of the increment and of the new latent
    assert_block_parity(lat - lat0, new_ref - lat0, what="latent increment")
    assert cosine(lat, new_ref) >= 0.999


def test_denoise_euler_fused_bit_exact():
    """The output projection's second pass applies the Euler update in its
    epilogue: the new latent equals latent + (sigma_next - sigma) v exactly,
    v being the velocity the step returns, the product rounded before the add
    (float32 arithmetic in numpy, which does not fuse)."""
    wl = TINY_DIT
    s = O.flowmatch_sigmas(8, 4.0)
    sig, sig_n = float(s[2]), float(s[3])
    mw = synth.model_weights(wl, seed=0, n_layers=2)
    cfg = dit.model_config_from(wl, 2)
    model = dit.DeviceModel(mw, dev())
    lat0 = synth.latent_input(wl, seed=1).to(dev()).contiguous()
    lat = lat0.clone()
    v = torch.empty_like(lat)
    dit.dit_denoise_step(cfg, model, lat, synth.text_input(wl, seed=1).to(dev()), wl.grid_h,
                         wl.grid_w, sig, sig_n, velocity_out=v)
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    dt = np.float32(sig_n) - np.float32(sig)
    want = (npf(lat0) + dt * npf(v)).astype(np.float32)
    np.testing.assert_array_equal(npf(lat), want)


def test_whole_loop_cuda_graph_matches_eager():
    """All 8 Euler steps of a small denoiser captured in one CUDA graph (the
    library allocates nothing and never synchronises, so the path captures);
    replaying it gives exactly the eager result."""
    wl = TINY_DIT
    mw = synth.model_weights(wl, seed=0, n_layers=2)
    cfg = dit.model_config_from(wl, 2)
    model = dit.DeviceModel(mw, dev())
    text = synth.text_input(wl, seed=1).to(dev())
    lat0 = synth.latent_input(wl, seed=1).to(dev())
    ws = dit.workspace(dit.dit_denoise_workspace_bytes(cfg, wl.grid_h, wl.grid_w, wl.n_txt), dev())
    s = dit.flowmatch_sigmas(8, 4.0)

    def loop(lat):
        for i in range(8):
            dit.dit_denoise_step(cfg, model, lat, text, wl.grid_h, wl.grid_w, s[i], s[i + 1], ws=ws)

    eager = lat0.clone()
    loop(eager)
    torch.cuda.synchronize()
    lat = lat0.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            loop(lat)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):          # replay twice from the same start
        lat.copy_(lat0)
        g.replay()
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    np.testing.assert_array_equal(npf(lat), npf(eager))


@pytest.mark.parametrize("name", ["ernie_full", "krea_gqa"])
def test_denoise_step_full_size_two_layers(name):
    """Full token count and width of the 36-layer ERNIE-shaped and 28-layer
    Krea-shaped denoisers, with 2 layers so the oracle finishes in seconds:
    conditioning, patch embedding, sequence assembly, RoPE tables, blocks,
    final norm, projection and Euler update are all exercised at size."""
    wl = synth.WORKLOADS[name]
    s = O.flowmatch_sigmas(8, 4.0)
    lat, v, new_ref, v_ref, lat0 = run_denoise(wl, 2, float(s[1]), float(s[2]))
    assert_block_parity(v, v_ref, what=f"{name} velocity")
    assert cosine(v, v_ref) >= 0.999
    assert cosine(lat, new_ref) >= 0.999
