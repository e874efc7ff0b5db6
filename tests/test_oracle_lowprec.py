"""Pins for the oracle's low-precision linears: the 256-point Hadamard
rotation, the e4m3 rounding and decoding, per-row coding and the W8A8 H256
linear ([ZFLOW] "From Python + CUDA to Pure Rust + Metal 4", section VII).
Library routines (scipy's Hadamard matrix, torch's float8_e4m3fn casts),
closed forms and error bounds; CPU only."""
import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import dit_oracle as O

F32 = np.float32
RNG = np.random.default_rng(4321)


def rnd(*shape, scale=1.0):
    return (RNG.standard_normal(shape) * scale).astype(F32)


def torch_e4m3(v):
    return torch.from_numpy(np.ascontiguousarray(v, dtype=F32)).to(torch.float8_e4m3fn).float().numpy()


# ------------------------------------------------------------- rotation
def test_fwht_matches_library_hadamard():
    H = scipy.linalg.hadamard(256).astype(np.float64) / 16.0
    x = rnd(3, 768)
    want = (x.astype(np.float64).reshape(3, 3, 256) @ H).reshape(3, 768)
    got = O.fwht256_rows(x)
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-5 * np.abs(want).max())


def test_fwht_basis_rows_are_hadamard_rows():
    H = scipy.linalg.hadamard(256).astype(F32) / F32(16)
    for i in (0, 1, 2, 77, 128, 255):
        e = np.zeros((1, 256), F32)
        e[0, i] = 1.0
        np.testing.assert_array_equal(O.fwht256_rows(e)[0], H[i])


def test_fwht_orthogonal_and_involution():
    x = rnd(4, 512)
    y = O.fwht256_rows(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)
    np.testing.assert_allclose(O.fwht256_rows(y), x, atol=1e-5)


def test_fwht_blocks_are_independent():
    x = rnd(2, 512)
    x2 = x.copy()
    x2[:, 256:] = rnd(2, 256)
    a, b = O.fwht256_rows(x), O.fwht256_rows(x2)
    np.testing.assert_array_equal(a[:, :256], b[:, :256])
    assert not np.array_equal(a[:, 256:], b[:, 256:])


def test_fwht_rejects_ragged_axis():
    with pytest.raises(ValueError):
        O.fwht256_rows(rnd(2, 300))


def test_rotation_rule():
    # (x H)(W H)^T = x W^T for the orthogonal H ([ZFLOW] section VII)
    x, w = rnd(5, 512), rnd(7, 512)
    lhs = O.fwht256_rows(x).astype(np.float64) @ O.fwht256_rows(w).astype(np.float64).T
    rhs = x.astype(np.float64) @ w.astype(np.float64).T
    np.testing.assert_allclose(lhs, rhs, atol=1e-4)


# ------------------------------------------------------------- e4m3
def test_e4m3_decode_table_matches_library():
    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = O.e4m3_decode_table()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert np.nanmax(got) == 448.0 and got[1] == 2.0 ** -9


def test_e4m3_round_worked_values():
    cases = {
        0.0: 0.0, 1.0: 1.0, 1.0625: 1.0,  # tie between 1 and 1.125: even mantissa 0
        1.1875: 1.25,                      # tie between 1.125 and 1.25: even mantissa 2
        2.0 ** -10: 0.0,                   # half the smallest subnormal: ties to 0
        3 * 2.0 ** -10: 2.0 ** -8,         # between 1 and 2 steps of 2^-9: even 2
        -3.3: -3.25, 0.017: 0.017578125,   # 0.017 = 8.704 steps of 2^-9 -> 9 steps
        448.0: 448.0, 460.0: 448.0, 470.0: 448.0, -1000.0: -448.0,  # saturated
        240.0: 240.0, 250.0: 256.0,
    }
    v = np.array(list(cases.keys()), F32)
    np.testing.assert_array_equal(O.e4m3_round(v), np.array(list(cases.values()), F32))


def test_e4m3_round_matches_library():
    grid = O.e4m3_decode_table()
    grid = np.unique(grid[~np.isnan(grid)]).astype(np.float64)
    mids = (grid[1:] + grid[:-1]) / 2          # exact ties
    v = np.concatenate([
        grid, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
        RNG.standard_normal(20000) * 2.0 ** RNG.integers(-12, 9, 20000),
    ]).astype(F32)
    v = v[np.abs(v) <= 448.0]
    np.testing.assert_array_equal(O.e4m3_round(v), torch_e4m3(v))


# ------------------------------------------------------------- coding
def test_quantize_rows_properties():
    y = rnd(6, 512) * np.array([1e-3, 1, 3, 50, 1e4, 0.2], F32)[:, None]
    y[3, :] = 0.0
    codes, scale = O.quantize_rows_e4m3(y)
    assert scale[3] == 0.0 and not codes[3].any()
    for r in (0, 1, 2, 4, 5):
        amax = np.abs(y[r]).max()
        assert scale[r] == F32(amax) / F32(448.0)
        j = np.abs(y[r]).argmax()
        assert abs(codes[r, j]) == 448.0
        assert np.abs(codes[r]).max() <= 448.0
        # half a step of the code's binade (3 mantissa bits), or of the subnormal step
        t = y[r].astype(np.float64) * (448.0 / np.float64(amax))
        half = np.maximum(np.ldexp(1.0, np.frexp(np.abs(t))[1] - 1 - 4), 2.0 ** -10)
        assert np.all(np.abs(codes[r] - t) <= half * (1 + 1e-6) + 1e-4)
    # every value is one code
    assert np.isin(codes, O.e4m3_decode_table()).all()


def test_w8a8_exact_on_hadamard_rows():
    # x = 1.75 h_j and w rows = 3.5 h_k with h the orthonormal Hadamard rows:
    # their rotations are 1.75 e_j and 3.5 e_k, coded exactly as 448 with the
    # exact scales 2^-8 and 2^-7; so y = 6.125 delta_jk exactly.
    H = scipy.linalg.hadamard(256).astype(F32) / F32(16)
    x = np.stack([F32(1.75) * H[5], F32(1.75) * H[200]])
    w = np.stack([F32(3.5) * H[k] for k in (5, 9, 200)])
    y = O.linear_w8a8_h256(x, w)
    np.testing.assert_array_equal(y, np.array([[6.125, 0, 0], [0, 0, 6.125]], F32))


def test_w8a8_error_within_coding_bound():
    x, w = rnd(8, 768), rnd(5, 768, scale=0.02)
    xr, wr = O.fwht256_rows(x).astype(np.float64), O.fwht256_rows(w).astype(np.float64)
    qx, sx = O.rotate_quantize(x)
    qw, sw = O.rotate_quantize(w)
    dx = qx * sx[:, None].astype(np.float64) - xr
    dw = qw * sw[:, None].astype(np.float64) - wr
    bound = np.abs(xr) @ np.abs(dw).T + np.abs(dx) @ np.abs(wr).T + np.abs(dx) @ np.abs(dw).T
    y = O.linear_w8a8_h256(x, w).astype(np.float64)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.all(np.abs(y - exact) <= bound * (1 + 1e-5) + 1e-6)
    # and each coded element is within the e4m3 half step (relative 2^-4)
    assert np.all(np.abs(dx) <= np.abs(xr) * 2.0 ** -4 + sx[:, None] * 2.0 ** -10 + 1e-12)
    rel = np.sqrt(np.mean((y - exact) ** 2) / np.mean(exact ** 2))
    assert rel < 0.06


def test_w8a8_sensitive_to_operand_orientation():
    # transposing the weight or skipping the rotation of one operand must fail
    x, w = rnd(4, 256), rnd(3, 256)
    y = O.linear_w8a8_h256(x, w)
    exact = x @ w.T
    qx, sx = O.quantize_rows_e4m3(x)            # unrotated activations
    qw, sw = O.rotate_quantize(w)
    wrong = (qx @ qw.T) * sx[:, None] * sw[None, :]
    assert np.abs(y - exact).max() < 0.2 * np.abs(exact).max()
    assert np.abs(wrong - exact).max() > 0.5 * np.abs(exact).max()


# ------------------------------------------------------------- block
def _small_block(fmt):
    cfg = O.BlockConfig(hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=768,
                        linear_format=fmt)
    w = {
        "w_qkv": rnd(768, 256, scale=0.02), "w_o": rnd(256, 256, scale=0.02),
        "w_gu": rnd(1536, 256, scale=0.02), "w_down": rnd(256, 768, scale=0.02),
        "q_g": 1 + rnd(64, scale=0.1), "q_b": rnd(64, scale=0.1),
        "k_g": 1 + rnd(64, scale=0.1), "k_b": rnd(64, scale=0.1),
    }
    return cfg, w


def test_w8a8_block_close_to_bf16_block_and_rows_agree():
    cfg8, w = _small_block("w8a8_h256")
    cfg16, _ = _small_block("bf16")
    n = 48
    x = rnd(n, 256)
    mod = rnd(6, 256, scale=0.5)
    ang = RNG.uniform(0, 6, (n, 32)).astype(F32)
    y8 = O.block_forward(cfg8, w, x, mod, ang)
    y16 = O.block_forward(cfg16, w, x, mod, ang)
    d8, d16 = y8 - x, y16 - x
    rel = np.sqrt(np.mean((d8 - d16) ** 2) / np.mean(d16 ** 2))
    assert 1e-4 < rel < 0.1
    rows = np.array([0, 7, 47])
    np.testing.assert_allclose(O.block_forward_rows(cfg8, w, x, mod, ang, rows), y8[rows],
                               atol=1e-5)


def test_w8a8_block_zero_gates_pass_residual():
    cfg, w = _small_block("w8a8_h256")
    x = rnd(16, 256)
    mod = rnd(6, 256)
    mod[2] = 0.0
    mod[5] = 0.0
    ang = RNG.uniform(0, 6, (16, 32)).astype(F32)
    np.testing.assert_array_equal(O.block_forward(cfg, w, x, mod, ang), x)
