"""Per-kernel GPU parity: each stage of the path, called through the C ABI,
against the oracle's function of the same name on the same seeded inputs.
Sizes span several tiles and a ragged tail."""
import numpy as np
import pytest
import torch

from gpu_common import bf16_normal, dev, npf, pair_major_tables
from oracle import dit_oracle as O

pytestmark = pytest.mark.gpu

dit = pytest.importorskip("diffusion_transformer_image_gb300.dit")

BF16_REL = 2.0 ** -8   # one bf16 rounding of the output: the unit roundoff of 8 significant bits


def _rms(a):
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


# ------------------------------------------------------------------ GEMM
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (130, 384, 128), (300, 512, 4096),
                                   (257, 128, 192), (1, 256, 256), (200, 320, 200)])
def test_linear_bf16(M, N, K):
    a = bf16_normal((M, K), f"lin_a{M}_{K}")
    w = bf16_normal((N, K), f"lin_w{N}_{K}", std=0.05)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev())
    dit.dit_linear(dit.DIT_EPI_BF16, a.to(dev()), w.to(dev()), out)
    ref = O.linear(npf(a), npf(w))
    got = npf(out)
    np.testing.assert_allclose(got, ref, rtol=BF16_REL, atol=1e-3 * _rms(ref))


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (200, 128, 4096), (129, 640, 256)])
def test_linear_f32_bias(M, N, K):
    a = bf16_normal((M, K), f"lb_a{M}_{K}")
    w = bf16_normal((N, K), f"lb_w{N}_{K}", std=0.05)
    b = bf16_normal((N,), f"lb_b{N}", std=0.5).float()
    out = torch.empty(M, N, dtype=torch.float32, device=dev())
    dit.dit_linear(dit.DIT_EPI_F32_BIAS, a.to(dev()), w.to(dev()), out, b.to(dev()))
    ref = O.linear(npf(a), npf(w), npf(b))
    np.testing.assert_allclose(npf(out), ref, rtol=1e-4, atol=1e-4 * _rms(ref))


@pytest.mark.parametrize("gated", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 256, 1024), (260, 100, 136)])
def test_linear_gated_residual(M, N, K, gated):
    a = bf16_normal((M, K), f"gr_a{M}_{K}")
    w = bf16_normal((N, K), f"gr_w{N}_{K}", std=0.05)
    x = bf16_normal((M, N), f"gr_x{M}_{N}").float()
    g = bf16_normal((N,), f"gr_g{N}", std=0.5).float() if gated else None
    xg = x.to(dev()).contiguous()
    dit.dit_linear(dit.DIT_EPI_RESIDUAL, a.to(dev()), w.to(dev()), xg,
                   None if g is None else g.to(dev()))
    ref = O.gated_residual(npf(x), None if g is None else npf(g), O.linear(npf(a), npf(w)))
    np.testing.assert_allclose(npf(xg), ref, rtol=1e-5, atol=1e-4 * _rms(ref))


@pytest.mark.parametrize("M,F,K", [(256, 128, 256), (300, 384, 512), (130, 768, 256)])
def test_linear_swiglu(M, F, K):
    a = bf16_normal((M, K), f"sw_a{M}_{K}")
    w = bf16_normal((2 * F, K), f"sw_w{F}_{K}", std=0.08)
    out = torch.empty(M, F, dtype=torch.bfloat16, device=dev())
    dit.dit_linear(dit.DIT_EPI_SWIGLU, a.to(dev()), w.to(dev()), out)
    gu = O.linear(npf(a), npf(w))
    ref = O.silu(gu[:, :F]) * gu[:, F:]
    np.testing.assert_allclose(npf(out), ref, rtol=BF16_REL, atol=1e-3 * _rms(ref))


# ------------------------------------------------------------ row kernels
@pytest.mark.parametrize("rows,H", [(37, 256), (130, 4096), (8, 6144), (5, 1024)])
def test_ln_modulate_adaln(rows, H):
    x = (bf16_normal((rows, H), f"ln_x{rows}_{H}", std=2.0).float() + 0.5)
    shift = bf16_normal((H,), f"ln_sh{H}", std=0.5).float()
    scale = bf16_normal((H,), f"ln_sc{H}", std=0.5).float()
    out = torch.empty(rows, H, dtype=torch.bfloat16, device=dev())
    dit.dit_ln_modulate(0, x.to(dev()), shift.to(dev()), scale.to(dev()), 1e-6, out)
    ref = O.modulate(O.layer_norm(npf(x), 1e-6), npf(shift), npf(scale))
    np.testing.assert_allclose(npf(out), ref, rtol=BF16_REL, atol=1e-4)


def test_ln_affine():
    rows, H = 69, 1024
    x = bf16_normal((rows, H), "lna_x").float()
    g = bf16_normal((H,), "lna_g", std=0.02, mean=1.0).float()
    b = bf16_normal((H,), "lna_b", std=0.02).float()
    out = torch.empty(rows, H, dtype=torch.bfloat16, device=dev())
    dit.dit_ln_modulate(1, x.to(dev()), g.to(dev()), b.to(dev()), 1e-6, out)
    ref = O.layer_norm(npf(x), 1e-6) * npf(g) + npf(b)
    np.testing.assert_allclose(npf(out), ref, rtol=BF16_REL, atol=1e-4)


@pytest.mark.parametrize("n", [4096 * 128, 1001, 3])
def test_euler_bit_exact(n):
    x = torch.randn(n, generator=torch.Generator().manual_seed(n))
    v = torch.randn(n, generator=torch.Generator().manual_seed(n + 1))
    s = O.flowmatch_sigmas(8, 4.0)
    xg = x.to(dev()).contiguous()
    dit.flowmatch_euler_step(xg, v.to(dev()), float(s[2]), float(s[3]))
    ref = O.euler_step(x.numpy(), v.numpy(), s[2], s[3])
    np.testing.assert_array_equal(npf(xg), ref)


def test_sigmas_host_match_oracle():
    np.testing.assert_array_equal(np.array(dit.flowmatch_sigmas(8, 4.0), np.float32),
                                  O.flowmatch_sigmas(8, 4.0))


@pytest.mark.parametrize("gh,gw,ntxt,axes", [(16, 16, 0, (16, 24, 24)), (64, 64, 256, (32, 48, 48)),
                                             (5, 7, 3, (32, 48, 48))])
def test_rope_table_grid(gh, gw, ntxt, axes):
    n, half = gh * gw + ntxt, sum(axes) // 2
    c = torch.empty(half, n, device=dev())
    s = torch.empty(half, n, device=dev())
    dit.dit_rope_table_grid(gh, gw, ntxt, axes, 256.0, c, s)
    ang = O.rope_angles_3d(O.position_ids(gh, gw, ntxt), axes, 256.0)   # [n, half]
    np.testing.assert_allclose(npf(c), np.cos(ang).T, atol=2e-6, rtol=0)
    np.testing.assert_allclose(npf(s), np.sin(ang).T, atol=2e-6, rtol=0)
    # the same table from explicit positions
    pos = torch.from_numpy(O.position_ids(gh, gw, ntxt)).to(dev())
    c2 = torch.empty_like(c)
    s2 = torch.empty_like(s)
    dit.dit_rope_table_pos(pos, axes, 256.0, c2, s2)
    assert torch.equal(c, c2) and torch.equal(s, s2)


def test_rope_table_vit():
    c = torch.empty(32, 5 + 32 * 32, device=dev())
    s = torch.empty_like(c)
    dit.dit_rope_table_vit(32, 32, 5, 64, 10000.0, c, s)
    ang = O.rope_angles_vit(32, 32, 5, 64)   # [n, half]
    np.testing.assert_allclose(npf(c), np.cos(ang).T, atol=2e-6, rtol=0)
    np.testing.assert_allclose(npf(s), np.sin(ang).T, atol=2e-6, rtol=0)


# ------------------------------------------------------- QKV + attention
QKV_CASES = {
    # name: hidden, nh, nkv, hd, layout, qk_norm, s_len, n_seqs
    "mha64": (256, 4, 4, 64, "interleaved", True, 256, 1),
    "gqa128_tail": (256, 6, 2, 128, "interleaved", True, 300, 1),
    "vit_seqs": (256, 4, 4, 64, "half", False, 133, 2),
    "odd_heads": (192, 3, 3, 64, "interleaved", True, 70, 1),
}


def _qkv_setup(case):
    H, nh, nkv, hd, layout, qkn, S, ns = QKV_CASES[case]
    n = S * ns
    cfg = dit.block_config(H, nh, nkv, hd, 256, layout, True, qkn)
    w = {"w_qkv": bf16_normal(((nh + 2 * nkv) * hd, H), f"q_w{case}", std=0.05)}
    if qkn:
        w["q_g"] = bf16_normal((hd,), f"q_qg{case}", std=0.1, mean=1.0).float()
        w["q_b"] = bf16_normal((hd,), f"q_qb{case}", std=0.1).float()
        w["k_g"] = bf16_normal((hd,), f"q_kg{case}", std=0.1, mean=1.0).float()
        w["k_b"] = bf16_normal((hd,), f"q_kb{case}", std=0.1).float()
    a = bf16_normal((n, H), f"q_a{case}")
    if layout == "half":
        side = int(np.ceil(np.sqrt(S)))
        ang = np.zeros((S, hd // 2), np.float32)
        full = O.rope_angles_vit(side, side, 0, hd)
        ang[:] = full[:S]
    else:
        pos = np.stack([np.arange(S) % 5, np.arange(S) // 7, np.arange(S) % 11], 1).astype(np.int32)
        ang = O.rope_angles_3d(pos, (16, 24, 24) if hd == 64 else (32, 48, 48), 256.0)
    ocfg = O.BlockConfig(H, nh, nkv, hd, 256, rope_layout=layout, qk_norm=qkn)
    return cfg, w, a, ang, ocfg, (H, nh, nkv, hd, S, ns)


@pytest.mark.parametrize("case", list(QKV_CASES))
def test_qkv_rope(case):
    cfg, w, a, ang, ocfg, (H, nh, nkv, hd, S, ns) = _qkv_setup(case)
    n = S * ns
    s_pad = (S + 7) // 8 * 8
    blk = dit.DeviceBlock(dict(w, w_o=w["w_qkv"], w_gu=w["w_qkv"], w_down=w["w_qkv"]), dev())
    rc, rs = pair_major_tables(ang)
    qk = torch.zeros(nh + nkv, n, hd, dtype=torch.bfloat16, device=dev())
    vt = torch.zeros(ns, nkv, hd, s_pad, dtype=torch.bfloat16, device=dev())
    dit.dit_qkv_rope(cfg, blk, a.to(dev()), rc, rs, qk, vt, n_seqs=ns)
    ow = {k: npf(v) for k, v in w.items()}
    q, k, v = O.qkv_heads(ocfg, npf(a), ow, np.tile(ang, (ns, 1)))
    gq = npf(qk)[:nh].transpose(1, 0, 2)      # head-major -> [n, nh, hd]
    gk = npf(qk)[nh:].transpose(1, 0, 2)
    gv = npf(vt)[..., :S].transpose(0, 3, 1, 2).reshape(n, nkv, hd)
    for got, ref in ((gq, q), (gk, k), (gv, v)):
        np.testing.assert_allclose(got, ref, rtol=BF16_REL, atol=2e-3 * _rms(ref))


ATTN_CASES = {
    # name: nh, nkv, hd, s_len, n_seqs, q_scale, growing keys
    "mha64_256": (4, 4, 64, 256, 1, 1.0, False),
    "gqa128_tail": (6, 2, 128, 300, 1, 1.0, False),
    "seqs_tail": (2, 1, 64, 133, 3, 1.0, False),
    "peaky_rescale": (2, 2, 128, 520, 1, 6.0, True),
    "single_block": (1, 1, 128, 77, 1, 2.0, False),
}


@pytest.mark.parametrize("case", list(ATTN_CASES))
def test_attention(case):
    nh, nkv, hd, S, ns, qs, grow = ATTN_CASES[case]
    n = S * ns
    s_pad = (S + 7) // 8 * 8
    q = bf16_normal((n, nh, hd), f"at_q{case}", std=qs)
    kf = bf16_normal((n, nkv, hd), f"at_k{case}").float()
    if grow:  # later keys larger: the running maximum keeps growing
        ramp = 1.0 + 3.0 * (torch.arange(n).float() % S) / S
        kf = kf * ramp[:, None, None]
    k = kf.to(torch.bfloat16)
    v = bf16_normal((n, nkv, hd), f"at_v{case}")
    qk = torch.cat([q.permute(1, 0, 2), k.permute(1, 0, 2)], 0).contiguous()  # head-major
    vt = torch.zeros(ns, nkv, hd, s_pad, dtype=torch.bfloat16)
    vt[..., :S] = v.reshape(ns, S, nkv, hd).permute(0, 2, 3, 1)
    o = torch.full((n, nh * hd), float("nan"), dtype=torch.bfloat16, device=dev())
    cfg = dit.block_config(256, nh, nkv, hd, 256)
    dit.dit_attention(cfg, qk.to(dev()), vt.to(dev()), o, n_seqs=ns)
    ref = O.attention(npf(q), npf(k), npf(v), nh, nkv, ns)
    got = npf(o)
    assert np.isfinite(got).all()
    rms = _rms(ref)
    err = np.abs(got - ref)
    rnd = np.abs(_bf16(ref) - ref)     # storing the exact output in bf16 alone
    print(f"attention {case}: max|err| {err.max() / rms:.4f} x RMS, bf16 output rounding "
          f"alone {rnd.max() / rms:.4f} x RMS, max|err| - rounding {(err - rnd).max() / rms:.4f} x RMS")
    # Element by element, the rounding the kernel does: one bf16 rounding of
    # the output (at most 2^-8 |o|, the unit roundoff of 8 significant bits)
    # and P rounded to bf16 before the PV product.  A relative error of at
    # most 2^-8 in every weight p_j moves o = sum p_j v_j / sum p_j by at most
    # 2 * 2^-8 * sum p_j |v_j| / sum p_j, i.e. 2^-7 times attention over |v|.
    p_bound = 2.0 ** -7 * O.attention(npf(q), npf(k), np.abs(npf(v)), nh, nkv, ns)
    bound = BF16_REL * np.abs(ref) + p_bound
    print(f"attention {case}: largest |err| / element bound {(err / bound).max():.3f}")
    assert np.all(err <= bound + 1e-3 * rms), (err - bound).max() / rms
    # The block bound, max|err| <= 2e-2 RMS(o), unless the bf16 rounding of
    # the exact output alone already exceeds it (heavy-tailed rows).
    assert err.max() <= max(2e-2 * rms, 1.25 * rnd.max() + 1e-3 * rms), (err.max() / rms, rnd.max() / rms)


def test_bounded_wait_reports_timeout_and_context_survives():
    assert dit.dit_last_device_error() == dit.DIT_OK
    dit.dit_set_wait_timeout_ns(2_000_000)      # 2 ms
    try:
        dit.dit_debug_stuck_wait()
        assert dit.dit_last_device_error() == dit.DIT_ETIMEOUT
        assert dit.dit_last_device_error() == dit.DIT_OK   # the word was cleared
    finally:
        dit.dit_set_wait_timeout_ns(2_000_000_000)
    # the context is still usable
    x = torch.ones(1024, device=dev())
    v = torch.ones(1024, device=dev())
    dit.flowmatch_euler_step(x, v, 1.0, 0.5)
    assert torch.all(x == 0.5)


def test_invalid_arguments_enqueue_nothing():
    cfg = dit.block_config(256, 4, 4, 96, 768)   # head_dim 96 is outside the kernel set
    x = torch.zeros(256, 256, device=dev())
    with pytest.raises(dit.DitError) as e:
        dit.dit_block_forward(cfg, None, x, None, x, x, ws=torch.zeros(256, dtype=torch.uint8, device=dev()))
    assert e.value.status in (dit.DIT_EUNSUPPORTED, dit.DIT_EINVAL)


def test_empty_inputs():
    """Zero rows or elements enqueue nothing and leave the buffers alone; an
    empty token sequence or an empty GEMM is rejected before any launch."""
    H = 1024
    x = torch.randn(4, H, device=dev())
    out = torch.full((4, H), 7.0, dtype=torch.bfloat16, device=dev())
    p = torch.zeros(H, device=dev())
    dit.dit_ln_modulate(0, x[:0], p, p, 1e-6, out[:0])
    xb = x.to(torch.bfloat16)
    codes = torch.full((4, H), 3, dtype=torch.uint8, device=dev())
    scales = torch.full((4,), 5.0, device=dev())
    dit.dit_rotate_quantize(xb[:0], codes[:0], scales[:0])
    dit.dit_ln_modulate_rotate_quantize(0, x[:0], p, p, 1e-6, codes[:0], scales[:0])
    v = torch.randn(16, device=dev())
    xe = torch.full((16,), 0.5, device=dev())
    dit.flowmatch_euler_step(xe[:0], v[:0], 1.0, 0.5)
    torch.cuda.synchronize()
    assert dit.dit_last_device_error() == dit.DIT_OK
    assert torch.all(out == 7.0) and torch.all(codes == 3) and torch.all(scales == 5.0)
    assert torch.all(xe == 0.5)
    with pytest.raises(dit.DitError) as e:
        dit.dit_linear(dit.DIT_EPI_BF16, xb[:0], xb, out[:0])
    assert e.value.status == dit.DIT_EINVAL
    cfg = dit.block_config(256, 4, 4, 64, 768)
    with pytest.raises(dit.DitError) as e:
        dit.dit_block_forward(cfg, None, x[:0, :256], None, x, x,
                              ws=torch.zeros(256, dtype=torch.uint8, device=dev()))
    assert e.value.status == dit.DIT_EINVAL


# ------------------------------------------------------------- variants
@pytest.mark.parametrize("rows,H,affine", [(37, 256, False), (130, 4096, False), (69, 1024, True)])
def test_rms_modulate(rows, H, affine):
    x = (bf16_normal((rows, H), f"rms_x{rows}_{H}", std=2.0).float() + 0.5)
    p0 = bf16_normal((H,), f"rms_p0{H}", std=0.5).float()
    p1 = bf16_normal((H,), f"rms_p1{H}", std=0.5).float()
    out = torch.empty(rows, H, dtype=torch.bfloat16, device=dev())
    dit.dit_ln_modulate(3 if affine else 2, x.to(dev()), p0.to(dev()), p1.to(dev()), 1e-6, out)
    n = O.rms_norm(npf(x), 1e-6)
    ref = n * npf(p0) + npf(p1) if affine else O.modulate(n, npf(p0), npf(p1))
    np.testing.assert_allclose(npf(out), ref, rtol=BF16_REL, atol=1e-4)


@pytest.mark.parametrize("M,F,K", [(256, 128, 256), (300, 384, 512)])
def test_linear_geglu(M, F, K):
    a = bf16_normal((M, K), f"gg_a{M}_{K}")
    w = bf16_normal((2 * F, K), f"gg_w{F}_{K}", std=0.3)   # large gates reach the clamps
    out = torch.empty(M, F, dtype=torch.bfloat16, device=dev())
    dit.dit_linear(dit.DIT_EPI_GEGLU, a.to(dev()), w.to(dev()), out)
    gu = O.linear(npf(a), npf(w))
    ref = O.gelu_tanh_clamped(gu[:, :F]) * gu[:, F:]
    np.testing.assert_allclose(npf(out), ref, rtol=BF16_REL, atol=1e-3 * _rms(ref))


@pytest.mark.parametrize("fn", ["tanh", "sigmoid"])
def test_linear_gated_residual_gate_functions(fn):
    M, N, K = 300, 256, 512
    a = bf16_normal((M, K), f"gf_a{fn}")
    w = bf16_normal((N, K), f"gf_w{fn}", std=0.05)
    x = bf16_normal((M, N), f"gf_x{fn}").float()
    g = bf16_normal((N,), f"gf_g{fn}", std=2.0).float()
    xg = x.to(dev()).contiguous()
    epi = dit.DIT_EPI_RESIDUAL_TANH if fn == "tanh" else dit.DIT_EPI_RESIDUAL_SIGMOID
    dit.dit_linear(epi, a.to(dev()), w.to(dev()), xg, g.to(dev()))
    ref = O.gated_residual(npf(x), O.gate_act(npf(g), fn), O.linear(npf(a), npf(w)))
    np.testing.assert_allclose(npf(xg), ref, rtol=1e-5, atol=1e-4 * _rms(ref))


@pytest.mark.parametrize("kind,order", [("rms", "norm_rope"), ("layer", "rope_norm"), ("rms", "rope_norm")])
@pytest.mark.parametrize("case", ["mha64", "gqa128_tail"])
def test_qkv_norm_variants(case, kind, order):
    cfg, w, a, ang, ocfg, (H, nh, nkv, hd, S, ns) = _qkv_setup(case)
    cfg.norm_kind = dit.NORM_KINDS[kind]
    cfg.rope_order = dit.ROPE_ORDERS[order]
    ocfg.norm_kind, ocfg.rope_order = kind, order
    n = S * ns
    s_pad = (S + 7) // 8 * 8
    blk = dit.DeviceBlock(dict(w, w_o=w["w_qkv"], w_gu=w["w_qkv"], w_down=w["w_qkv"]), dev())
    rc, rs = pair_major_tables(ang)
    qk = torch.zeros(nh + nkv, n, hd, dtype=torch.bfloat16, device=dev())
    vt = torch.zeros(ns, nkv, hd, s_pad, dtype=torch.bfloat16, device=dev())
    dit.dit_qkv_rope(cfg, blk, a.to(dev()), rc, rs, qk, vt, n_seqs=ns)
    q, k, _ = O.qkv_heads(ocfg, npf(a), {kk: npf(vv) for kk, vv in w.items()}, np.tile(ang, (ns, 1)))
    for got, ref in ((npf(qk)[:nh].transpose(1, 0, 2), q), (npf(qk)[nh:].transpose(1, 0, 2), k)):
        np.testing.assert_allclose(got, ref, rtol=BF16_REL, atol=2e-3 * _rms(ref))
