"""The W8A8 format with the H256 rotation on the GPU against the oracle
([ZFLOW] "From Python + CUDA to Pure Rust + Metal 4", section VII).

Coding from bf16 rows is bit-exact (same fp32 butterflies in the same order,
same divisions and roundings).  Coding fused behind the norm may differ by one
e4m3 step where the norm's fp32 statistics differ in the last bits.  The e4m3
GEMM is compared with the float64 sum of the decoded code products, also at
the full-size shapes.  Small blocks and a small denoise step in the W8A8
format meet the per-block criterion against the oracle's W8A8 block; the
full-size blocks meet a bound derived from how far bf16 storage alone moves
the format's codes (see that test)."""
import dataclasses

import numpy as np
import pytest
import torch

from diffusion_transformer_image_gb300 import synth
from gpu_common import (assert_block_parity, bf16_storage_rows, cosine, dev, max_err_vs_rms, npf,
                        oracle_angles, oracle_block_config, oracle_weights, pair_major_tables)
from oracle import dit_oracle as O
from test_gpu_block import (SMALL_BLOCKS, conditioning_pair, run_block_gpu, run_denoise,
                            sample_rows, TINY_DIT)

pytestmark = pytest.mark.gpu

dit = pytest.importorskip("diffusion_transformer_image_gb300.dit")

TABLE = O.e4m3_decode_table()


def decode(codes: torch.Tensor) -> np.ndarray:
    return TABLE[codes.cpu().numpy().astype(np.int64)]


def w8(wl):
    return dataclasses.replace(wl, linear_format="w8a8_h256")


def rows_input(rows, K, seed):
    """bf16 rows with scales from 1e-3 to 1e3, one zero row and one row with
    an outlier column."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g)
    scale = 10.0 ** torch.empty(rows, 1).uniform_(-3, 3, generator=g)
    x = x * scale
    x[rows // 2] = 0.0
    if rows > 2:
        x[1, 7] = 500.0 * float(scale[1])
    return x.to(torch.bfloat16)


# ------------------------------------------------------------- coding kernels
# K = 1024 and 3072 take 32 values per thread of the TMA-ring kernel, 2048
# and up in steps of 2048 take 64, the rest the warp-per-block kernel.
@pytest.mark.parametrize("rows,K", [(1, 256), (37, 768), (50, 3072), (130, 4096), (70, 6144),
                                    (9, 12288), (3, 16384)])
def test_rotate_quantize_bit_exact(rows, K):
    x = rows_input(rows, K, seed=rows + K)
    codes, scales = dit.dit_rotate_quantize(x.to(dev()))
    torch.cuda.synchronize()
    ref_codes, ref_scales = O.rotate_quantize(x.float().numpy())
    np.testing.assert_array_equal(npf(scales), ref_scales)
    np.testing.assert_array_equal(decode(codes), ref_codes)


def test_rotate_quantize_extreme_scales():
    """Rows scaled from 2^-120 to 2^100 on top of their own scales: codes and
    scales bit-identical to the oracle's from tiny to huge rows, including a
    row whose rotated values reach the subnormal range (the rotation's 1/16
    is one exact multiplication of every value, as in the oracle; moving it
    to the row scale would change such rows)."""
    base = rows_input(8, 4096, seed=11).float()
    f = torch.tensor([2.0 ** -100, 2.0 ** 100, 1.0, 2.0 ** -60, 2.0 ** 60, 2.0 ** -120, 3.0, 2.0 ** 90])
    x = (base * f[:, None]).to(torch.bfloat16)
    for K in (4096, 3072):   # 64 and 32 values per thread
        xs = x[:, :K].contiguous()
        codes, scales = dit.dit_rotate_quantize(xs.to(dev()))
        torch.cuda.synchronize()
        ref_codes, ref_scales = O.rotate_quantize(xs.float().numpy())
        np.testing.assert_array_equal(npf(scales), ref_scales)
        np.testing.assert_array_equal(decode(codes), ref_codes)


def test_rotate_quantize_strided_rows():
    x = rows_input(20, 1024, seed=5)
    big = torch.zeros(20, 1024 + 64, dtype=torch.bfloat16)
    big[:, :1024] = x
    codes = torch.full((20, 1024 + 32), 0x55, dtype=torch.uint8, device=dev())
    scales = torch.empty(20, device=dev())
    xg = big.to(dev())
    st = dit.lib.dit_rotate_quantize(dit._ptr(xg), xg.stride(0), 20, 1024, dit._ptr(codes),
                                     codes.stride(0), dit._ptr(scales), dit._stream())
    assert st == dit.DIT_OK
    torch.cuda.synchronize()
    ref_codes, ref_scales = O.rotate_quantize(x.float().numpy())
    np.testing.assert_array_equal(decode(codes[:, :1024]), ref_codes)
    np.testing.assert_array_equal(npf(scales), ref_scales)
    assert (codes[:, 1024:] == 0x55).all()  # the row padding is left alone


def _step(t):
    a = np.abs(t.astype(np.float64))
    e = np.maximum(np.frexp(a)[1] - 1, -6)
    return np.ldexp(1.0, e - 3)


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("H", [256, 4096])
def test_ln_modulate_rotate_quantize(mode, H):
    rows = 70
    x = synth.normal((rows, H), "lnq_x", 3 + mode, std=2.0, mean=0.5)
    p0 = synth.normal((H,), "lnq_p0", 4, std=0.5)
    p1 = synth.normal((H,), "lnq_p1", 5, std=0.5)
    codes = torch.empty(rows, H, dtype=torch.uint8, device=dev())
    scales = torch.empty(rows, device=dev())
    dit.dit_ln_modulate_rotate_quantize(mode, x.to(dev()), p0.to(dev()), p1.to(dev()), 1e-6,
                                        codes, scales)
    torch.cuda.synchronize()
    n = O.norm(npf(x), 1e-6, "rms" if mode & 2 else "layer")
    a = n * npf(p0) + npf(p1) if mode & 1 else O.modulate(n, npf(p0), npf(p1))
    y = O.fwht256_rows(a)
    ref_codes, ref_scales = O.quantize_rows_e4m3(y)
    np.testing.assert_allclose(npf(scales), ref_scales, rtol=2e-6)
    got = decode(codes)
    t = y.astype(np.float64) * (448.0 / np.abs(y).max(axis=1, keepdims=True))
    # each code is a grid neighbour of the exact target, and nearly all are
    # the oracle's code (the norm's statistics differ in the last bits only)
    assert np.all(np.abs(got - t) <= _step(t) + 1e-9)
    assert np.mean(got != ref_codes) < 2e-3


# ------------------------------------------------------------- e4m3 GEMM
def random_codes(rows, K, seed):
    """e4m3 codes with exponent fields 4..9 (|value| 2^-3 .. 7.5), random
    signs and mantissas, 5 % zeros."""
    g = torch.Generator().manual_seed(seed)
    e = torch.randint(4, 10, (rows, K), generator=g)
    m = torch.randint(0, 8, (rows, K), generator=g)
    s = torch.randint(0, 2, (rows, K), generator=g)
    c = (s << 7) | (e << 3) | m
    c[torch.rand(rows, K, generator=g) < 0.05] = 0
    return c.to(torch.uint8)


def e4m3_reference(a, sa, w, sw):
    A, W = decode(a).astype(np.float64), decode(w).astype(np.float64)
    sa64, sw64 = npf(sa).astype(np.float64), npf(sw).astype(np.float64)
    y = (A @ W.T) * sa64[:, None] * sw64[None, :]
    absy = (np.abs(A) @ np.abs(W).T) * sa64[:, None] * sw64[None, :]
    return y, absy


# fp32 accumulation of products that are exact: a relative bound on the sum
# of |products|, far below any coding or indexing slip (those move outputs
# by whole code steps, >= 1/16 of a term)
ACC_RTOL = 1e-5


@pytest.mark.parametrize("epi", ["bf16", "f32_bias", "residual", "residual_tanh",
                                 "residual_sigmoid"])
def test_linear_e4m3_plain_epilogues(epi):
    M, N, K = 300, 384, 1024
    a, w = random_codes(M, K, 1), random_codes(N, K, 2)
    g = torch.Generator().manual_seed(3)
    sa = torch.rand(M, generator=g) * 0.02 + 0.005
    sw = torch.rand(N, generator=g) * 0.02 + 0.005
    y, absy = e4m3_reference(a, sa, w, sw)
    vec = torch.randn(N, generator=g)
    kind = {"bf16": dit.DIT_EPI_BF16, "f32_bias": dit.DIT_EPI_F32_BIAS,
            "residual": dit.DIT_EPI_RESIDUAL, "residual_tanh": dit.DIT_EPI_RESIDUAL_TANH,
            "residual_sigmoid": dit.DIT_EPI_RESIDUAL_SIGMOID}[epi]
    if epi == "bf16":
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev())
        dit.dit_linear_e4m3(kind, a.to(dev()), sa.to(dev()), w.to(dev()), sw.to(dev()), out)
        ref, tol = y, ACC_RTOL * absy + 2.0 ** -8 * np.abs(y)
    else:
        x0 = torch.randn(M, N, generator=g)
        out = x0.clone().to(dev())
        dit.dit_linear_e4m3(kind, a.to(dev()), sa.to(dev()), w.to(dev()), sw.to(dev()), out,
                            bias_or_gate=vec.to(dev()))
        v = npf(vec).astype(np.float64)
        if epi == "f32_bias":
            ref, tol = y + v[None, :], ACC_RTOL * absy + 1e-6
        else:
            fn = {"residual": "identity", "residual_tanh": "tanh",
                  "residual_sigmoid": "sigmoid"}[epi]
            gate = O.gate_act(npf(vec), fn).astype(np.float64)
            ref = npf(x0) + gate[None, :] * y
            tol = ACC_RTOL * absy * np.abs(gate)[None, :] + 1e-6 * (1 + np.abs(ref))
    torch.cuda.synchronize()
    got = npf(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol), float(np.max(np.abs(got - ref) / (tol + 1e-30)))


@pytest.mark.parametrize("glu", ["silu", "gelu_tanh"])
def test_linear_e4m3_glu(glu):
    M, F, K = 260, 256, 768
    a, w = random_codes(M, K, 4), random_codes(2 * F, K, 5)
    g = torch.Generator().manual_seed(6)
    sa = torch.rand(M, generator=g) * 0.02 + 0.005
    sw = torch.rand(2 * F, generator=g) * 0.02 + 0.005
    y, absy = e4m3_reference(a, sa, w, sw)
    out = torch.empty(M, F, dtype=torch.bfloat16, device=dev())
    kind = dit.DIT_EPI_SWIGLU if glu == "silu" else dit.DIT_EPI_GEGLU
    dit.dit_linear_e4m3(kind, a.to(dev()), sa.to(dev()), w.to(dev()), sw.to(dev()), out)
    torch.cuda.synchronize()
    cfg = O.BlockConfig(hidden=K, n_heads=1, n_kv_heads=1, head_dim=64, ffn=F, glu=glu)
    ref = O.glu(cfg, y.astype(np.float32)).astype(np.float64)
    # the accumulator bound carried through the activation (slope <= 1.2) and
    # the product with up, plus the bf16 store
    gate, up = y[:, :F], y[:, F:]
    dacc = ACC_RTOL * absy
    tol = 1.2 * dacc[:, :F] * np.abs(up) + dacc[:, F:] * (np.abs(gate) + 1) + \
        2.0 ** -8 * np.abs(ref) + 1e-6
    got = npf(out).astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol), float(np.max(np.abs(got - ref) / tol))


@pytest.mark.parametrize("shape", ["down", "gate_up"])
def test_linear_e4m3_full_size_sampled_rows(shape):
    """The ERNIE-shaped down (K = 12288, residual epilogue) and gate/up
    (N = 2 x 12288, SwiGLU) projections at 4352 rows: many tiles per
    persistent CTA and long K; sampled rows against float64."""
    M = 4352
    if shape == "down":
        N, K, rowsW = 4096, 12288, 4096
    else:
        N, K, rowsW = 12288, 4096, 2 * 12288
    a, w = random_codes(M, K, 7), random_codes(rowsW, K, 8)
    g = torch.Generator().manual_seed(9)
    sa = torch.rand(M, generator=g) * 0.002 + 0.0005
    sw = torch.rand(rowsW, generator=g) * 0.002 + 0.0005
    rows = sample_rows(M)
    y, absy = e4m3_reference(a[rows], sa[rows], w, sw)
    if shape == "down":
        gate = torch.randn(N, generator=g)
        x0 = torch.randn(M, N, generator=g)
        out = x0.clone().to(dev())
        dit.dit_linear_e4m3(dit.DIT_EPI_RESIDUAL, a.to(dev()), sa.to(dev()), w.to(dev()),
                            sw.to(dev()), out, bias_or_gate=gate.to(dev()))
        gv = npf(gate).astype(np.float64)
        ref = npf(x0)[rows] + gv[None, :] * y
        tol = ACC_RTOL * absy * np.abs(gv)[None, :] + 1e-6 * (1 + np.abs(ref))
    else:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev())
        dit.dit_linear_e4m3(dit.DIT_EPI_SWIGLU, a.to(dev()), sa.to(dev()), w.to(dev()),
                            sw.to(dev()), out)
        gate_v, up = y[:, :N], y[:, N:]
        ref = (O.silu(gate_v.astype(np.float32)).astype(np.float64)) * up
        dacc = ACC_RTOL * absy
        tol = 1.2 * dacc[:, :N] * np.abs(up) + dacc[:, N:] * (np.abs(gate_v) + 1) + \
            2.0 ** -8 * np.abs(ref) + 1e-6
    torch.cuda.synchronize()
    got = npf(out)[rows].astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol), float(np.max(np.abs(got - ref) / tol))


@pytest.mark.parametrize("case", ["mha64", "gqa128_tail", "vit_seqs"])
def test_qkv_rope_e4m3(case):
    """The QKV projection on codes with its fused qk-norm + RoPE epilogue; the
    activation codes come from bf16 rows, so both sides code identically."""
    from test_gpu_kernels import BF16_REL, _qkv_setup, _rms
    cfg, w, a, ang, ocfg, (H, nh, nkv, hd, S, ns) = _qkv_setup(case)
    cfg.linear_format = dit.LINEAR_FORMATS["w8a8_h256"]
    ocfg.linear_format = "w8a8_h256"
    n = S * ns
    s_pad = (S + 7) // 8 * 8
    blk = dit.DeviceBlock(dict(w, w_o=w["w_qkv"], w_gu=w["w_qkv"], w_down=w["w_qkv"]), dev(),
                          "w8a8_h256")
    codes, sa = dit.dit_rotate_quantize(a.to(dev()))
    rc, rs = pair_major_tables(ang)
    qk = torch.zeros(nh + nkv, n, hd, dtype=torch.bfloat16, device=dev())
    vt = torch.zeros(ns, nkv, hd, s_pad, dtype=torch.bfloat16, device=dev())
    dit.dit_qkv_rope_e4m3(cfg, blk, codes, sa, rc, rs, qk, vt, n_seqs=ns)
    torch.cuda.synchronize()
    q, k, v = O.qkv_heads(ocfg, npf(a), {kk: npf(vv) for kk, vv in w.items()},
                          np.tile(ang, (ns, 1)))
    gq = npf(qk)[:nh].transpose(1, 0, 2)
    gk = npf(qk)[nh:].transpose(1, 0, 2)
    gv = npf(vt)[..., :S].transpose(0, 3, 1, 2).reshape(n, nkv, hd)
    for got, ref in ((gq, q), (gk, k), (gv, v)):
        np.testing.assert_allclose(got, ref, rtol=BF16_REL, atol=2e-3 * _rms(ref))


def test_w8a8_invalid_arguments():
    x = torch.zeros(4, 300, dtype=torch.bfloat16, device=dev())
    with pytest.raises(dit.DitError) as e:
        dit.dit_rotate_quantize(x)
    assert e.value.status == dit.DIT_EINVAL
    cfg = dit.block_config(320, 5, 5, 64, 768, linear_format="w8a8_h256")  # 320 % 256 != 0
    assert dit.dit_block_workspace_bytes(cfg, 64) == 0
    wl = w8(synth.WORKLOADS["tiny_block"])
    w = synth.block_weights(wl, 0, seed=0)
    blk = dit.DeviceBlock(w, dev())          # bf16 weights, no scales
    cfg = dit.block_config_from(wl)
    xg = torch.zeros(wl.n_tokens, wl.hidden, device=dev())
    c = torch.zeros(wl.n_tokens, wl.head_dim // 2, device=dev())
    with pytest.raises(dit.DitError) as e:
        dit.dit_block_forward(cfg, blk, xg, torch.zeros(6, wl.hidden, device=dev()), c, c)
    assert e.value.status == dit.DIT_EINVAL


# ------------------------------------------------------------- blocks
@pytest.mark.parametrize("name", list(SMALL_BLOCKS))
def test_block_w8a8_small(name):
    """Every output of a small block in the W8A8 format against the oracle's
    W8A8 block; the bf16 block differs from both by the coding error."""
    wl = w8(SMALL_BLOCKS[name])
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = (None, None)
    if wl.adaln:
        mod_g = synth.modulation_input(wl, seed=1)
        mod_o = npf(mod_g)
    got = run_block_gpu(wl, w, x, mod_g)
    cfg, ow, ang = oracle_block_config(wl), oracle_weights(w), oracle_angles(wl)
    ref = O.block_forward(cfg, ow, npf(x), mod_o, ang, wl.n_seqs)
    rel = assert_block_parity(got, ref, what=f"{name} w8a8")
    ref16 = O.block_forward(dataclasses.replace(cfg, linear_format="bf16"), ow, npf(x), mod_o,
                            ang, wl.n_seqs)
    e16, rms = max_err_vs_rms(ref16, ref)
    print(f"{name}: gpu vs oracle w8a8 {rel:.3e} RMS; bf16 vs w8a8 oracle {e16 / rms:.3e} RMS")
    assert rel < 0.5 * e16 / rms


@pytest.mark.parametrize("name", ["ernie_block", "krea_gqa"])
def test_block_w8a8_full_size_sampled_rows(name):
    """Full size, modulation from the timestep MLP at t = 0.5, 48 sampled rows.
    At this size a perturbation far below bf16 resolution flips some e4m3
    codes, and each flip moves its element by a whole code step: the oracle's
    own evaluation with the GPU's bf16 storage of q/k/v, o and h differs from
    the fp32 oracle by about 4 % (ERNIE-shaped) and 13 % (Krea-shaped) of RMS
    at the worst element, so the per-block 2e-2 bound cannot hold for any
    implementation of the format that stores those in bf16.  The bound is
    derived from that arithmetic instead: the GPU's distance from the oracle
    may be at most 1.5 x the distance of that bf16-storage evaluation (which
    leaves out the GPU's other last-bit differences: norm statistics,
    accumulation order, the attention's bf16 P), in the worst element and in
    RMS."""
    wl = w8(synth.WORKLOADS[name])
    w = synth.block_weights(wl, 0, seed=0)
    x = synth.residual_input(wl, seed=1)
    mod_g, mod_o = conditioning_pair(wl, wl.t_block)
    rows = sample_rows(wl.n_tokens)
    got = run_block_gpu(wl, w, x, mod_g)[rows]
    cfg, ow, ang = oracle_block_config(wl), oracle_weights(w), oracle_angles(wl)
    ref = O.block_forward_rows(cfg, ow, npf(x), mod_o, ang, rows)
    sim = bf16_storage_rows(cfg, ow, npf(x), mod_o, ang, rows)
    e_gpu, rms = max_err_vs_rms(got, ref)
    e_sim, _ = max_err_vs_rms(sim, ref)
    r_gpu = float(np.sqrt(np.mean((got - ref) ** 2))) / rms
    r_sim = float(np.sqrt(np.mean((sim - ref) ** 2))) / rms
    print(f"{name} w8a8: gpu max {e_gpu / rms:.4f} rms {r_gpu:.5f}; "
          f"bf16-storage oracle max {e_sim / rms:.4f} rms {r_sim:.5f}")
    assert np.isfinite(got).all()
    assert e_gpu <= 1.5 * e_sim + 1e-3 * rms
    assert r_gpu <= 1.5 * r_sim + 1e-4
    assert cosine(got, ref) >= 0.999


@pytest.mark.parametrize("step", [0, 5])
def test_denoise_step_w8a8_tiny(step):
    s = O.flowmatch_sigmas(8, 4.0)
    lat, v, new_ref, v_ref, lat0 = run_denoise(w8(TINY_DIT), 2, float(s[step]),
                                               float(s[step + 1]))
    assert_block_parity(v, v_ref, what="w8a8 velocity")
    assert cosine(lat, new_ref) >= 0.999
