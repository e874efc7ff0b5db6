"""Pins for the CPU oracle: closed forms, brute force, invariants and the
pages' worked values.  Each test is chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a
swapped chunk) fails it.  CPU only."""
import math
import os

import numpy as np
import pytest

from oracle import dit_oracle as O

F32 = np.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def rnd(*shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(F32)


# ---------------------------------------------------------------- linear
def test_linear_selects_input_features():
    # W[out, in] one-hot: y[:, o] must equal x[:, sel[o]] (catches W vs W^T)
    x = rnd(5, 7)
    sel = [3, 0, 6]
    w = np.zeros((3, 7), F32)
    for o, i in enumerate(sel):
        w[o, i] = 1.0
    b = np.array([0.5, -1.0, 2.0], F32)
    y = O.linear(x, w, b)
    assert y.shape == (5, 3)
    for o, i in enumerate(sel):
        np.testing.assert_array_equal(y[:, o], x[:, i] + b[o])


def test_linear_brute_force():
    x, w = rnd(4, 9), rnd(6, 9)
    y = O.linear(x, w)
    for r in range(4):
        for o in range(6):
            s = 0.0
            for k in range(9):
                s += float(x[r, k]) * float(w[o, k])
            assert abs(y[r, o] - s) <= 1e-5 * (1 + abs(s))


# ---------------------------------------------------------------- silu
def test_silu_closed_forms():
    assert O.silu(np.array([0.0], F32))[0] == 0.0
    # sigmoid(ln 3) = 3/4
    x = math.log(3.0)
    assert abs(O.silu(np.array([x], F32))[0] - 0.75 * x) < 1e-6
    big = O.silu(np.array([40.0, -40.0], F32))
    assert abs(big[0] - 40.0) < 1e-5 and abs(big[1]) < 1e-12


# ---------------------------------------------------------------- norm
def test_layer_norm_hand_example():
    y = O.layer_norm(np.array([[1, 2, 3, 4]], F32), 0.0)
    # mean 2.5, biased variance 1.25
    np.testing.assert_allclose(y[0], np.array([-1.5, -0.5, 0.5, 1.5]) / math.sqrt(1.25), rtol=1e-6)


def test_layer_norm_moments_and_invariance():
    x = rnd(16, 256, scale=3.0) + 5.0
    y = O.layer_norm(x, 1e-6)
    assert np.abs(y.mean(axis=1)).max() < 1e-5
    assert np.abs(y.var(axis=1) - 1.0).max() < 1e-4
    # affine invariance of the input: LN(a x + c) == LN(x) for a > 0
    np.testing.assert_allclose(O.layer_norm(2.0 * x - 7.0, 1e-6), y, atol=2e-5)


def test_modulate_plus_one():
    xn = rnd(3, 8)
    shift, scale = rnd(8), rnd(8)
    # scale = -1 removes the normalised input entirely: output is the shift
    np.testing.assert_array_equal(O.modulate(xn, shift, -np.ones(8, F32)), np.broadcast_to(shift, (3, 8)))
    np.testing.assert_array_equal(O.modulate(xn, np.zeros(8, F32), np.zeros(8, F32)), xn)
    np.testing.assert_allclose(O.modulate(xn, shift, scale), xn + xn * scale + shift, rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------- positions
def test_position_ids_golden():
    rows = [list(map(int, ln.split())) for ln in open(os.path.join(GOLDEN, "position_ids_2x3_txt2.txt"))
            if ln.strip() and not ln.startswith("#")]
    np.testing.assert_array_equal(O.position_ids(2, 3, 2), np.array(rows, np.int32))


def test_position_ids_text_first_is_a_permutation():
    a = O.position_ids(4, 5, 3, image_first=True)
    b = O.position_ids(4, 5, 3, image_first=False)
    np.testing.assert_array_equal(np.concatenate([a[20:], a[:20]]), b)


# ---------------------------------------------------------------- rope
def test_rope_angles_closed_form_theta256():
    # theta = 256 = 2^8.  Axis of size 16: inv_freq_j = 2^(-8*2j/16) = 2^-j.
    # Axis of size 24: inv_freq_j = 2^(-2j/3).
    pos = np.array([[3, 5, 7], [0, 1, 2]], np.int32)
    ang = O.rope_angles_3d(pos, (16, 24, 24), 256.0)
    assert ang.shape == (2, 32)
    for r in range(2):
        for j in range(8):
            assert ang[r, j] == F32(pos[r, 0] * 2.0 ** -j)
        for j in range(12):
            np.testing.assert_allclose(ang[r, 8 + j], pos[r, 1] * 2.0 ** (-2 * j / 3), rtol=1e-6)
            np.testing.assert_allclose(ang[r, 20 + j], pos[r, 2] * 2.0 ** (-2 * j / 3), rtol=1e-6)


def test_rope_apply_quarter_turn():
    ang = np.array([[math.pi / 2, 0.0]], F32)
    x = np.array([[1.0, 0.0, 2.0, 3.0]], F32)
    yi = O.rope_apply(x, ang, "interleaved")       # pairs (0,1), (2,3)
    np.testing.assert_allclose(yi, [[0.0, 1.0, 2.0, 3.0]], atol=1e-7)
    yh = O.rope_apply(x, ang, "half")              # pairs (0,2), (1,3)
    np.testing.assert_allclose(yh, [[-2.0, 0.0, 1.0, 3.0]], atol=1e-6)


@pytest.mark.parametrize("layout", ["interleaved", "half"])
def test_rope_norm_preserved_and_identity_at_zero(layout):
    x = rnd(2, 10, 64)
    ang = rnd(10, 32, scale=20.0)
    y = O.rope_apply(x, ang, layout)
    if layout == "interleaved":
        nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
        ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    else:
        nx = x[..., :32] ** 2 + x[..., 32:] ** 2
        ny = y[..., :32] ** 2 + y[..., 32:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=2e-5, atol=1e-6)
    np.testing.assert_array_equal(O.rope_apply(x, np.zeros((10, 32), F32), layout), x)


def test_rope_relative_position():
    # <R(p) q, R(p') k> depends only on p - p' on every axis
    axes = (16, 24, 24)
    q, k = rnd(64), rnd(64)
    p1 = np.array([[3, 10, 4], [1, 2, 9]], np.int32)
    off = np.array([[7, -2, 5]], np.int32)

    def dot(p):
        a = O.rope_angles_3d(p, axes, 256.0)
        rq = O.rope_apply(q[None], a[:1], "interleaved")[0]
        rk = O.rope_apply(k[None], a[1:], "interleaved")[0]
        return float(np.dot(rq.astype(np.float64), rk.astype(np.float64)))

    assert abs(dot(p1) - dot(p1 + off)) < 1e-4


def test_rope_vit_table_prefix_unrotated():
    ang = O.rope_angles_vit(4, 4, 5, 64)
    assert ang.shape == (21, 32)
    assert np.all(ang[:5] == 0)
    # patch (r=2, c=3): first quarter r*w_k, second quarter c*w_k, w_0 = 1
    t = 5 + 2 * 4 + 3
    assert ang[t, 0] == 2.0 and ang[t, 16] == 3.0
    np.testing.assert_allclose(ang[t, 8], 2.0 * 10000.0 ** (-8 / 16), rtol=1e-6)


# ---------------------------------------------------------------- attention
def brute_attention(q, k, v, nh, nkv):
    n, _, d = q.shape
    out = np.zeros((n, nh, d))
    for h in range(nh):
        g = h // (nh // nkv)
        for i in range(n):
            s = [sum(float(q[i, h, c]) * float(k[j, g, c]) for c in range(d)) / math.sqrt(d)
                 for j in range(n)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for c in range(d):
                out[i, h, c] = sum(e[j] / z * float(v[j, g, c]) for j in range(n))
    return out.reshape(n, nh * d)


def test_attention_brute_force_gqa():
    q, k, v = rnd(6, 4, 8), rnd(6, 2, 8), rnd(6, 2, 8)
    np.testing.assert_allclose(O.attention(q, k, v, 4, 2), brute_attention(q, k, v, 4, 2), rtol=1e-5, atol=1e-6)


def test_attention_identical_keys_give_mean_of_v():
    q, v = rnd(5, 1, 8), rnd(5, 1, 8)
    k = np.repeat(rnd(1, 1, 8), 5, axis=0)
    o = O.attention(q, k, v, 1, 1)
    np.testing.assert_allclose(o, np.repeat(v.mean(axis=0), 5, axis=0), rtol=1e-5, atol=1e-6)


def test_attention_huge_logit_copies_row():
    d = 8
    k = np.zeros((5, 1, d), F32)
    k[3, 0, 0] = 1.0
    q = np.zeros((5, 1, d), F32)
    q[:, 0, 0] = 1e4
    v = rnd(5, 1, d)
    np.testing.assert_allclose(O.attention(q, k, v, 1, 1), np.repeat(v[3], 5, axis=0), rtol=1e-6)


def test_attention_gqa_equals_repeated_mha():
    q, k, v = rnd(7, 6, 8), rnd(7, 2, 8), rnd(7, 2, 8)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    np.testing.assert_allclose(O.attention(q, k, v, 6, 2), O.attention(q, kr, vr, 6, 6), rtol=1e-6)


def test_attention_sequences_are_independent():
    q, k, v = rnd(10, 2, 8), rnd(10, 2, 8), rnd(10, 2, 8)
    both = O.attention(q, k, v, 2, 2, n_seqs=2)
    np.testing.assert_allclose(both[:5], O.attention(q[:5], k[:5], v[:5], 2, 2), rtol=1e-6)
    np.testing.assert_allclose(both[5:], O.attention(q[5:], k[5:], v[5:], 2, 2), rtol=1e-6)


# ---------------------------------------------------------------- timestep
def test_timestep_embedding_closed_forms():
    e0 = O.timestep_embedding(0.0, 256)
    np.testing.assert_array_equal(e0, np.concatenate([np.ones(128), np.zeros(128)]).astype(F32))
    t = 500.0
    e = O.timestep_embedding(t, 256)
    # j = 0: w = 1 -> cos(t), sin(t); j = 64: w = 10000^-0.5 = 0.01
    assert abs(e[0] - math.cos(t)) < 1e-4 and abs(e[128] - math.sin(t)) < 1e-4
    assert abs(e[64] - math.cos(5.0)) < 1e-5 and abs(e[192] - math.sin(5.0)) < 1e-5


# ---------------------------------------------------------------- scheduler
def test_sigmas_match_exponential_time_shift():
    s = O.flowmatch_sigmas(8, 4.0)
    assert s.shape == (9,) and s[0] == 1.0 and s[-1] == 0.0
    mu = math.log(4.0)
    for i in range(8):
        t = 1.0 - i / 8
        ref = math.exp(mu) / (math.exp(mu) + (1.0 / t - 1.0) ** 1.0)
        assert abs(s[i] - ref) < 1e-6
    assert np.all(np.diff(s) < 0)
    # shift 1 leaves the linear grid
    np.testing.assert_allclose(O.flowmatch_sigmas(8, 1.0), 1.0 - np.arange(9) / 8, atol=1e-7)


def test_euler_constant_velocity_integrates_to_minus_v():
    s = O.flowmatch_sigmas(8, 4.0)
    x0, v = rnd(32, 16), rnd(32, 16)
    x = x0
    for i in range(8):
        x = O.euler_step(x, v, s[i], s[i + 1])
    np.testing.assert_allclose(x, x0 - v, atol=1e-5)
    np.testing.assert_array_equal(O.euler_step(x0, v, 0.5, 0.5), x0)


# ---------------------------------------------------------------- block
def tiny_cfg(**kw):
    c = dict(hidden=64, n_heads=2, n_kv_heads=2, head_dim=32, ffn=96)
    c.update(kw)
    return O.BlockConfig(**c)


def tiny_weights(cfg, seed=0):
    r = np.random.default_rng(seed)
    nq = (cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim
    w = {
        "w_qkv": (r.standard_normal((nq, cfg.hidden)) * 0.2).astype(F32),
        "w_o": (r.standard_normal((cfg.hidden, cfg.n_heads * cfg.head_dim)) * 0.2).astype(F32),
        "w_gu": (r.standard_normal((2 * cfg.ffn, cfg.hidden)) * 0.2).astype(F32),
        "w_down": (r.standard_normal((cfg.hidden, cfg.ffn)) * 0.2).astype(F32),
        "q_g": (1 + 0.1 * r.standard_normal(cfg.head_dim)).astype(F32),
        "q_b": (0.1 * r.standard_normal(cfg.head_dim)).astype(F32),
        "k_g": (1 + 0.1 * r.standard_normal(cfg.head_dim)).astype(F32),
        "k_b": (0.1 * r.standard_normal(cfg.head_dim)).astype(F32),
        "ln1_g": (1 + 0.1 * r.standard_normal(cfg.hidden)).astype(F32),
        "ln1_b": (0.1 * r.standard_normal(cfg.hidden)).astype(F32),
        "ln2_g": (1 + 0.1 * r.standard_normal(cfg.hidden)).astype(F32),
        "ln2_b": (0.1 * r.standard_normal(cfg.hidden)).astype(F32),
    }
    return w


AXES = (8, 12, 12)


def tiny_inputs(n_img_h=3, n_img_w=4, n_txt=3, hidden=64, seed=5):
    r = np.random.default_rng(seed)
    x = r.standard_normal((n_img_h * n_img_w + n_txt, hidden)).astype(F32)
    mod = (0.5 * r.standard_normal((6, hidden))).astype(F32)
    pos = O.position_ids(n_img_h, n_img_w, n_txt)
    return x, mod, pos


def test_block_zero_gates_is_identity():
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    x, mod, pos = tiny_inputs()
    mod[2] = 0.0
    mod[5] = 0.0
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    np.testing.assert_array_equal(O.block_forward(cfg, w, x, mod, ang), x)


def test_block_chunk_order():
    # gate1 = 0: the attention branch is off, so shift1/scale1 cannot matter,
    # while shift2/scale2 must.  A wrong chunk index breaks one of the two.
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    x, mod, pos = tiny_inputs()
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    mod[2] = 0.0
    base = O.block_forward(cfg, w, x, mod, ang)
    m2 = mod.copy()
    m2[0] += 1.0
    m2[1] += 1.0
    np.testing.assert_array_equal(O.block_forward(cfg, w, x, m2, ang), base)
    m3 = mod.copy()
    m3[3] += 1.0
    assert np.abs(O.block_forward(cfg, w, x, m3, ang) - base).max() > 1e-3


def test_block_swiglu_gate_first():
    # scale2 = -1 makes the FFN input equal shift2 on every row.  With shift2 =
    # e_0, gate rows reading feature 0 with weight -100 and up rows with
    # weight 1, silu(-100) * 1 ~ 0: the FFN adds nothing.  Swapped halves
    # would give silu(1) * (-100).
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    w["w_gu"][:] = 0.0
    w["w_gu"][: cfg.ffn, 0] = -100.0
    w["w_gu"][cfg.ffn:, 0] = 1.0
    x, mod, pos = tiny_inputs()
    mod[2] = 0.0          # attention branch off
    mod[3] = 0.0
    mod[3, 0] = 1.0       # shift2 = e_0
    mod[4] = -1.0         # scale2 = -1
    mod[5] = 1.0
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    np.testing.assert_allclose(O.block_forward(cfg, w, x, mod, ang), x, atol=1e-6)


def test_block_position_offset_invariance():
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    x, mod, pos = tiny_inputs()
    a = O.block_forward(cfg, w, x, mod, O.rope_angles_3d(pos, AXES, 256.0))
    b = O.block_forward(cfg, w, x, mod, O.rope_angles_3d(pos + np.array([5, 3, 2], np.int32), AXES, 256.0))
    np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-4)


def test_block_token_permutation_equivariance():
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    x, mod, pos = tiny_inputs()
    perm = np.random.default_rng(3).permutation(x.shape[0])
    a = O.block_forward(cfg, w, x, mod, O.rope_angles_3d(pos, AXES, 256.0))
    b = O.block_forward(cfg, w, x[perm], mod, O.rope_angles_3d(pos[perm], AXES, 256.0))
    np.testing.assert_allclose(b, a[perm], rtol=1e-5, atol=1e-5)


def test_qk_norm_applied_before_rope():
    # Undo the rotation of the returned q: what is left must be exactly
    # LN(q_raw) * g + b, which has per-head mean b.mean() when g = 1.
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    w["q_g"][:] = 1.0
    w["q_b"][:] = 0.0
    x, mod, pos = tiny_inputs()
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    a = O.modulate(O.layer_norm(x, cfg.ln_eps), mod[0], mod[1])
    q, k, v = O.qkv_heads(cfg, a, w, ang)
    qu = O.rope_apply(np.swapaxes(q, 0, 1), -ang, "interleaved")
    assert np.abs(qu.mean(axis=-1)).max() < 1e-5
    assert np.abs(qu.var(axis=-1) - 1.0).max() < 1e-3
    # the rotated q itself is not zero-mean (so the order is observable)
    assert np.abs(q.mean(axis=-1)).max() > 1e-2


def test_vit_block_plain_residual_and_sequences():
    cfg = tiny_cfg(adaln=False, qk_norm=False, rope_layout="half")
    w = tiny_weights(cfg)
    r = np.random.default_rng(9)
    s_len = 2 + 9
    x = r.standard_normal((2 * s_len, 64)).astype(F32)
    ang = O.rope_angles_vit(3, 3, 2, 32)
    both = O.block_forward(cfg, w, x, None, ang, n_seqs=2)
    one = O.block_forward(cfg, w, x[:s_len], None, ang, n_seqs=1)
    np.testing.assert_allclose(both[:s_len], one, rtol=1e-5, atol=1e-5)


def test_final_layer_chunk_order():
    # fin = [scale, shift]: scale = -1 makes the projected input the shift row
    r = np.random.default_rng(2)
    x = r.standard_normal((6, 16)).astype(F32)
    shift = r.standard_normal(16).astype(F32)
    fin = np.stack([-np.ones(16, F32), shift])
    w, b = r.standard_normal((4, 16)).astype(F32), r.standard_normal(4).astype(F32)
    out = O.final_layer(x, fin, w, b, 1e-6)
    np.testing.assert_allclose(out, np.repeat((shift @ w.T + b)[None], 6, axis=0), rtol=1e-5)


def test_denoise_step_tiny_runs_and_zero_dt_is_identity():
    cfg = tiny_cfg()
    mc = O.ModelConfig(block=cfg, n_layers=2, latent_channels=8, t_dim=16, rope_axes=AXES)
    r = np.random.default_rng(4)
    h = cfg.hidden
    mw = {
        "patch_w": r.standard_normal((h, 8)).astype(F32) * 0.1, "patch_b": np.zeros(h, F32),
        "t_w1": r.standard_normal((h, 16)).astype(F32) * 0.1, "t_b1": np.zeros(h, F32),
        "t_w2": r.standard_normal((h, h)).astype(F32) * 0.1, "t_b2": np.zeros(h, F32),
        "mod_w": r.standard_normal((6 * h, h)).astype(F32) * 0.1, "mod_b": np.zeros(6 * h, F32),
        "fin_w": r.standard_normal((2 * h, h)).astype(F32) * 0.1, "fin_b": np.zeros(2 * h, F32),
        "out_w": r.standard_normal((8, h)).astype(F32) * 0.1, "out_b": np.zeros(8, F32),
        "layers": [tiny_weights(cfg, s) for s in range(2)],
    }
    lat = r.standard_normal((12, 8)).astype(F32)
    txt = r.standard_normal((3, h)).astype(F32)
    new, v = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.8, 0.7, return_velocity=True)
    assert np.isfinite(v).all() and v.shape == (12, 8)
    np.testing.assert_allclose(new, lat + F32(F32(0.7) - F32(0.8)) * v, rtol=1e-6, atol=1e-6)
    same = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.8, 0.8)
    np.testing.assert_array_equal(same, lat)


def test_block_attention_branch_closed_form():
    # scale1 = -1 makes every row of the attention input equal shift1, so all
    # value rows are equal and attention returns that value row whatever the
    # scores: out = x + gate1 * ((shift1 Wv^T) Wo^T).  The FFN is off (gate2 = 0).
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    x, mod, pos = tiny_inputs()
    mod[1] = -1.0
    mod[5] = 0.0
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    hd = cfg.n_heads * cfg.head_dim
    wv = w["w_qkv"][2 * hd:]
    branch = (mod[0].astype(np.float64) @ wv.T.astype(np.float64)) @ w["w_o"].T.astype(np.float64)
    expect = x + mod[2] * branch[None, :]
    np.testing.assert_allclose(O.block_forward(cfg, w, x, mod, ang), expect, rtol=1e-5, atol=1e-5)


def test_attention_rows_matches_attention():
    q, k, v = rnd(9, 4, 8), rnd(9, 2, 8), rnd(9, 2, 8)
    rows = np.array([0, 4, 8, 3])
    np.testing.assert_allclose(O.attention_rows(q[rows], k, v, 4, 2), O.attention(q, k, v, 4, 2)[rows],
                               rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("adaln", [True, False])
def test_block_forward_rows_matches_block_forward(adaln):
    cfg = tiny_cfg(adaln=adaln, qk_norm=adaln)
    w = tiny_weights(cfg)
    x, mod, pos = tiny_inputs()
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    rows = np.array([1, 14, 0, 7])
    full = O.block_forward(cfg, w, x, mod if adaln else None, ang)
    np.testing.assert_allclose(O.block_forward_rows(cfg, w, x, mod if adaln else None, ang, rows),
                               full[rows], rtol=1e-5, atol=1e-5)


# ------------------------------------------------ variants of the block
def test_rms_norm_hand_example_and_scale():
    y = O.rms_norm(np.array([[1, 2, 3, 4]], F32), 0.0)
    np.testing.assert_allclose(y[0], np.array([1, 2, 3, 4]) / math.sqrt(7.5), rtol=1e-6)
    x = rnd(8, 64) + 3.0
    r = O.rms_norm(x, 0.0)
    np.testing.assert_allclose((r.astype(np.float64) ** 2).mean(axis=1), 1.0, rtol=1e-5)
    np.testing.assert_allclose(O.rms_norm(-2.5 * x, 0.0), -r, rtol=1e-5, atol=1e-6)
    # unlike LayerNorm, a constant offset is not removed
    assert np.abs(O.rms_norm(x, 1e-6).mean(axis=1)).min() > 0.5


def test_gelu_tanh_clamped_closed_forms():
    g = lambda v: float(O.gelu_tanh_clamped(np.array([v], F32))[0])
    assert g(0.0) == 0.0
    # GELU(1) by the tanh form: 0.5 (1 + tanh(0.7978845608 * 1.044715))
    assert abs(g(1.0) - 0.5 * (1 + math.tanh(0.7978845608 * 1.044715))) < 1e-6
    # odd part: gelu(x) - gelu(-x) = x exactly for the tanh form
    for v in (0.3, 1.7, 4.0):
        assert abs(g(v) - g(-v) - v) < 1e-5
    # close to the exact x Phi(x) (the tanh form's error is below 1e-3)
    for v in np.linspace(-6, 6, 49):
        exact = 0.5 * v * (1 + math.erf(v / math.sqrt(2)))
        assert abs(g(float(v)) - exact) < 1e-3
    # the argument clamp: tanh saturates, large inputs pass through, large
    # negative ones vanish; the output clamp at the half-precision maximum
    assert g(30.0) == 30.0 and abs(g(-30.0)) < 1e-12
    assert g(1e5) == 65504.0 and abs(g(-1e5)) < 1e-12


def test_gate_functions():
    g = np.array([0.0, math.log(3.0), math.atanh(0.5)], F32)
    np.testing.assert_array_equal(O.gate_act(g, "identity"), g)
    t = O.gate_act(g, "tanh")
    assert t[0] == 0.0 and abs(t[2] - 0.5) < 1e-6
    s = O.gate_act(g, "sigmoid")
    assert s[0] == 0.5 and abs(s[1] - 0.75) < 1e-6


def test_block_sigmoid_gate_at_zero_is_half_identity_gate():
    # sigmoid(0) = 1/2: a block with sigmoid gates and zero gate inputs equals
    # the identity-gate block with gates of exactly 1/2.
    cfg_s = tiny_cfg(gate_fn="sigmoid")
    cfg_i = tiny_cfg()
    w = tiny_weights(cfg_s)
    x, mod, pos = tiny_inputs()
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    m0 = mod.copy()
    m0[2] = 0.0
    m0[5] = 0.0
    mh = mod.copy()
    mh[2] = 0.5
    mh[5] = 0.5
    np.testing.assert_array_equal(O.block_forward(cfg_s, w, x, m0, ang), O.block_forward(cfg_i, w, x, mh, ang))
    # tanh(0) = 0: zero gates still give the identity
    np.testing.assert_array_equal(O.block_forward(tiny_cfg(gate_fn="tanh"), w, x, m0, ang), x)


def test_rope_norm_order():
    w_cfg = tiny_cfg()
    w = tiny_weights(w_cfg)
    x, mod, pos = tiny_inputs()
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    a = O.modulate(O.layer_norm(x, 1e-6), mod[0], mod[1])
    w1 = dict(w)
    w1["q_g"] = np.ones_like(w["q_g"])
    w1["q_b"] = np.zeros_like(w["q_b"])
    # LayerNorm after RoPE: the returned q is itself zero-mean, unit-variance
    q, _, _ = O.qkv_heads(tiny_cfg(rope_order="rope_norm"), a, w1, ang)
    assert np.abs(q.mean(axis=-1)).max() < 1e-5 and np.abs(q.var(axis=-1) - 1).max() < 1e-3
    # RMSNorm commutes with a rotation (norms are preserved) when g = 1, b = 0
    q1, k1, _ = O.qkv_heads(tiny_cfg(norm_kind="rms"), a, w1 | {"k_g": w1["q_g"], "k_b": w1["q_b"]}, ang)
    q2, k2, _ = O.qkv_heads(tiny_cfg(norm_kind="rms", rope_order="rope_norm"), a,
                            w1 | {"k_g": w1["q_g"], "k_b": w1["q_b"]}, ang)
    np.testing.assert_allclose(q1, q2, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(k1, k2, rtol=1e-4, atol=1e-5)
    # with a non-uniform gain the two orders differ
    q3, _, _ = O.qkv_heads(tiny_cfg(norm_kind="rms", rope_order="rope_norm"), a, w, ang)
    q4, _, _ = O.qkv_heads(tiny_cfg(norm_kind="rms"), a, w, ang)
    assert np.abs(q3 - q4).max() > 1e-2


def test_block_geglu_gate_first():
    # as the SwiGLU test: gate rows read feature 0 with weight -100, so the
    # clamped GELU of the gate is ~0 and the FFN adds nothing
    cfg = tiny_cfg(glu="gelu_tanh")
    w = tiny_weights(cfg)
    w["w_gu"][:] = 0.0
    w["w_gu"][: cfg.ffn, 0] = -100.0
    w["w_gu"][cfg.ffn:, 0] = 1.0
    x, mod, pos = tiny_inputs()
    mod[2] = 0.0
    mod[3] = 0.0
    mod[3, 0] = 1.0
    mod[4] = -1.0
    mod[5] = 1.0
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    np.testing.assert_allclose(O.block_forward(cfg, w, x, mod, ang), x, atol=1e-6)
    # and with the halves swapped the FFN is active
    w["w_gu"][: cfg.ffn, 0] = 1.0
    w["w_gu"][cfg.ffn:, 0] = -100.0
    assert np.abs(O.block_forward(cfg, w, x, mod, ang) - x).max() > 1.0


def test_ernie_variant_block_invariants():
    # With RoPE before the qk-norm, relative-position invariance needs unit
    # gains and zero biases (a per-dimension gain after the rotation would
    # break it); RMSNorm then divides each rotated vector by its own length.
    cfg = tiny_cfg(norm_kind="rms", glu="gelu_tanh", rope_order="rope_norm")
    w = tiny_weights(cfg)
    for n in ("q", "k"):
        w[n + "_g"] = np.ones_like(w[n + "_g"])
        w[n + "_b"] = np.zeros_like(w[n + "_b"])
    x, mod, pos = tiny_inputs()
    ang = O.rope_angles_3d(pos, AXES, 256.0)
    a = O.block_forward(cfg, w, x, mod, ang)
    b = O.block_forward(cfg, w, x, mod, O.rope_angles_3d(pos + np.array([4, 1, 3], np.int32), AXES, 256.0))
    np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-4)
    rows = np.array([2, 0, 9])
    np.testing.assert_allclose(O.block_forward_rows(cfg, w, x, mod, ang, rows), a[rows], rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------------- conditioning
def _silu64(x):
    return x / (1.0 + math.exp(-x))


def _cond_weights(h, t_dim, sel, a, c, bm, b1=None, b2=None):
    """Hand-built time MLP and modulation heads whose outputs have closed
    forms: W1 row i picks sinusoid entry sel[i] times a[i]; W2 is diagonal
    c; modulation row (chunk k, column i) picks temb[i] times (k + 1), bias
    bm; the final head row (chunk k, column i) picks temb[i] times -(k + 1)."""
    w1 = np.zeros((h, t_dim), F32)
    for i, j in enumerate(sel):
        w1[i, j] = a[i]
    w2 = np.diag(np.asarray(c, F32))
    mw = np.zeros((6 * h, h), F32)
    fw = np.zeros((2 * h, h), F32)
    for k in range(6):
        for i in range(h):
            mw[k * h + i, i] = k + 1
    for k in range(2):
        for i in range(h):
            fw[k * h + i, i] = -(k + 1)
    return {"t_w1": w1, "t_b1": np.zeros(h, F32) if b1 is None else b1,
            "t_w2": w2, "t_b2": np.zeros(h, F32) if b2 is None else b2,
            "mod_w": mw, "mod_b": bm, "fin_w": fw, "fin_b": np.zeros(2 * h, F32)}


def test_conditioning_closed_form():
    # [ERNIE] section IV: the six adaLN chunks [shift1, scale1, gate1, shift2,
    # scale2, gate2] come from one H -> 6H linear of SiLU(temb), chunk k being
    # output rows [kH, (k+1)H); temb = W2 SiLU(W1 e + b1) + b2 with e the
    # sinusoid of T = 1000 sigma ([ZFLOW] section IV).  With one-hot weights
    # every output has a closed form: at sigma = 0.5, T = 500 and the
    # sinusoid entries 0 and 4 (t_dim 8, half 4: w_0 = 1) are cos 500 and
    # sin 500.  A missing SiLU (either one), T = sigma, a transposed [6H]
    # reshape or a swapped W1/W2 each changes some entry.
    h, td = 4, 8
    sel = [0, 4, 1, 5]                       # cos(T), sin(T), cos(T w_1), sin(T w_1)
    a = [2.0, -3.0, 1.5, 0.5]
    c = [1.0, 0.5, -2.0, 3.0]
    b1 = np.array([0.25, -0.5, 0.0, 1.0], F32)
    b2 = np.array([-0.75, 0.5, 0.125, 0.0], F32)
    bm = np.arange(6 * h, dtype=F32) * F32(0.01)
    mw = _cond_weights(h, td, sel, a, c, bm, b1, b2)
    sigma = 0.5
    mod, fin = O.conditioning(mw, sigma, td, 1000.0)
    assert mod.shape == (6, h) and fin.shape == (2, h)
    T = 1000.0 * sigma
    w1 = 10000.0 ** (-1 / 4)
    e = {0: math.cos(T), 4: math.sin(T), 1: math.cos(T * w1), 5: math.sin(T * w1)}
    temb = [c[i] * _silu64(a[i] * e[sel[i]] + float(b1[i])) + float(b2[i]) for i in range(h)]
    st = [_silu64(t) for t in temb]
    for k in range(6):
        for i in range(h):
            want = (k + 1) * st[i] + float(bm[k * h + i])
            assert abs(mod[k, i] - want) <= 2e-5 * (1 + abs(want)), (k, i, mod[k, i], want)
    for k in range(2):
        for i in range(h):
            want = -(k + 1) * st[i]
            assert abs(fin[k, i] - want) <= 2e-5 * (1 + abs(want)), (k, i, fin[k, i], want)


def test_conditioning_sigma_zero_feeds_cos_ones():
    # sigma = 0 gives T = 0 and the sinusoid [1 ... 1, 0 ... 0] (cosine half
    # first): a W1 row summing the cosine half sees t_dim / 2, a row summing
    # the sine half sees 0, whatever t_scale is.
    h, td = 2, 16
    mw = _cond_weights(h, td, [0, 0], [0.0, 0.0], [1.0, 1.0], np.zeros(6 * h, F32))
    mw["t_w1"] = np.zeros((h, td), F32)
    mw["t_w1"][0, : td // 2] = 0.25
    mw["t_w1"][1, td // 2:] = 1.0
    mod, _ = O.conditioning(mw, 0.0, td, 1000.0)
    temb = [_silu64(0.25 * td / 2), _silu64(0.0)]
    for i in range(h):
        assert abs(mod[0, i] - _silu64(temb[i])) <= 1e-6


# ---------------------------------------------------------------- step composition
def _step_model(cfg, seed=4, n_layers=2, c_lat=8, td=16, gates_off=False):
    r = np.random.default_rng(seed)
    h = cfg.hidden
    mw = {
        "patch_w": r.standard_normal((h, c_lat)).astype(F32) * 0.3,
        "patch_b": r.standard_normal(h).astype(F32) * 0.1,
        "t_w1": r.standard_normal((h, td)).astype(F32) * 0.1, "t_b1": np.zeros(h, F32),
        "t_w2": r.standard_normal((h, h)).astype(F32) * 0.1, "t_b2": np.zeros(h, F32),
        "mod_w": r.standard_normal((6 * h, h)).astype(F32) * 0.3,
        "mod_b": r.standard_normal(6 * h).astype(F32) * 0.3,
        "fin_w": r.standard_normal((2 * h, h)).astype(F32) * 0.3,
        "fin_b": r.standard_normal(2 * h).astype(F32) * 0.3,
        "out_w": r.standard_normal((c_lat, h)).astype(F32) * 0.3,
        "out_b": r.standard_normal(c_lat).astype(F32) * 0.1,
        "layers": [tiny_weights(cfg, s) for s in range(n_layers)],
    }
    if gates_off:  # gate1 = gate2 = 0: chunks 2 and 5 of the modulation
        for k in (2, 5):
            mw["mod_w"][k * h:(k + 1) * h] = 0.0
            mw["mod_b"][k * h:(k + 1) * h] = 0.0
    mc = O.ModelConfig(block=cfg, n_layers=n_layers, latent_channels=c_lat, t_dim=td,
                       rope_axes=AXES)
    return mc, mw


def test_denoise_step_zero_gates_is_head_then_tail():
    # With both gates zero every block is the identity ([ERNIE] section IV,
    # gated residuals), so the velocity is the final layer applied to the
    # patch embedding of the latent: the image rows of the joint sequence are
    # the patch-embedded latent, and the final layer reads those rows only
    # (the text must not matter).  Reading the text rows, or putting the text
    # first, fails this.
    cfg = tiny_cfg()
    mc, mw = _step_model(cfg, gates_off=True)
    r = np.random.default_rng(9)
    lat = r.standard_normal((12, 8)).astype(F32)
    txt = r.standard_normal((3, cfg.hidden)).astype(F32)
    _, v = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.8, 0.7, return_velocity=True)
    _, fin = O.conditioning(mw, 0.8, mc.t_dim, mc.t_scale)
    want = O.final_layer(O.linear(lat, mw["patch_w"], mw["patch_b"]), fin, mw["out_w"],
                         mw["out_b"], cfg.ln_eps)
    np.testing.assert_allclose(v, want, rtol=1e-5, atol=1e-5)
    _, v2 = O.denoise_step(mc, mw, lat, 5 * txt + 1, 3, 4, 0.8, 0.7, return_velocity=True)
    np.testing.assert_array_equal(v2, v)


def test_denoise_step_final_scale_minus_one_gives_shift_rows():
    # fin = [scale, shift] ([ERNIE] section V, Bug 4): a final head whose
    # weight is zero and whose bias is [-1 ... -1, s] makes every normed image
    # row s, so every velocity row is s Wout^T + bout, whatever the latent,
    # the text and the layers do.  A swapped chunk order fails.
    cfg = tiny_cfg()
    mc, mw = _step_model(cfg)
    h = cfg.hidden
    s = np.random.default_rng(3).standard_normal(h).astype(F32)
    mw["fin_w"][:] = 0.0
    mw["fin_b"] = np.concatenate([-np.ones(h, F32), s])
    r = np.random.default_rng(10)
    lat = r.standard_normal((12, 8)).astype(F32)
    txt = r.standard_normal((3, h)).astype(F32)
    _, v = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.6, 0.5, return_velocity=True)
    want = np.repeat((s @ mw["out_w"].T + mw["out_b"])[None], 12, axis=0)
    np.testing.assert_allclose(v, want, rtol=1e-5, atol=1e-5)


def test_denoise_step_text_reaches_image_rows_through_attention():
    # With the gates on, the text rows take part in the joint attention, so
    # changing the text changes the velocity of the image rows; and the
    # velocity depends on sigma through the modulation (T = 1000 sigma).
    cfg = tiny_cfg()
    mc, mw = _step_model(cfg)
    r = np.random.default_rng(11)
    lat = r.standard_normal((12, 8)).astype(F32)
    txt = r.standard_normal((3, cfg.hidden)).astype(F32)
    _, v = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.8, 0.7, return_velocity=True)
    _, v_txt = O.denoise_step(mc, mw, lat, txt[::-1].copy(), 3, 4, 0.8, 0.7,
                              return_velocity=True)
    _, v_sig = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.3, 0.2, return_velocity=True)
    assert np.abs(v_txt - v).max() > 1e-3
    assert np.abs(v_sig - v).max() > 1e-3


def test_denoise_step_equals_its_stages():
    # The step is its stages in the pages' order: conditioning at sigma,
    # patch embedding of the latent, [image rows; text rows], positions
    # (n_txt, h, w) / (j, 0, 0), the layers, the final layer on the image
    # rows, the Euler update ([ERNIE] section IV; [ZFLOW] section IV).
    cfg = tiny_cfg()
    mc, mw = _step_model(cfg)
    r = np.random.default_rng(12)
    lat = r.standard_normal((12, 8)).astype(F32)
    txt = r.standard_normal((3, cfg.hidden)).astype(F32)
    new, v = O.denoise_step(mc, mw, lat, txt, 3, 4, 0.8, 0.7, return_velocity=True)
    mod, fin = O.conditioning(mw, 0.8, mc.t_dim, mc.t_scale)
    x = np.concatenate([O.linear(lat, mw["patch_w"], mw["patch_b"]), txt])
    ang = O.rope_angles_3d(O.position_ids(3, 4, 3), AXES, 256.0)
    for lw in mw["layers"]:
        x = O.block_forward(cfg, lw, x, mod, ang)
    want_v = O.final_layer(x[:12], fin, mw["out_w"], mw["out_b"], cfg.ln_eps)
    np.testing.assert_array_equal(v, want_v)
    np.testing.assert_array_equal(new, O.euler_step(lat, want_v, 0.8, 0.7))
