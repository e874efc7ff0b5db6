"""CPU checks of the C ABI: the library loads, exports every entry point its
header declares, and rejects bad arguments on the host without touching a
GPU.  Builds libdit.so first when it is missing (nvcc cross-compiles)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dit.h")


@pytest.fixture(scope="module")
def dit():
    from diffusion_transformer_image_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from diffusion_transformer_image_gb300 import dit as d
    return d


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("dit_block_forward", "dit_denoise_step", "flowmatch_euler_step"):
        assert n in names


def test_library_exports_every_declared_symbol(dit):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(dit.lib, n), n
    assert sorted(dit.EXPORTED) == names


def test_sigmas_on_host_match_oracle(dit):
    from oracle import dit_oracle as O
    np.testing.assert_array_equal(np.array(dit.flowmatch_sigmas(8, 4.0), np.float32),
                                  O.flowmatch_sigmas(8, 4.0))
    np.testing.assert_array_equal(np.array(dit.flowmatch_sigmas(3, 1.0), np.float32),
                                  O.flowmatch_sigmas(3, 1.0))


def test_host_argument_checks(dit):
    cfg = dit.block_config(4096, 32, 32, 128, 12288)
    assert dit.lib.dit_block_forward(None, None, None, 0, 1, None, None, None, None, 0, None) == dit.DIT_EINVAL
    bad = dit.block_config(4096, 32, 32, 96, 12288)
    assert dit.lib.dit_block_workspace_bytes(ctypes.byref(bad), 4352, 1) == 0
    gqa_bad = dit.block_config(4096, 32, 5, 128, 12288)
    assert dit.lib.dit_block_forward(ctypes.byref(gqa_bad), None, None, 1, 1, None, None, None,
                                     None, 0, None) == dit.DIT_EUNSUPPORTED
    assert dit.lib.flowmatch_euler_step(ctypes.c_void_p(8), ctypes.c_void_p(16), 16, 1.0, 0.5,
                                        None) == dit.DIT_EINVAL   # misaligned x
    assert dit.lib.flowmatch_sigmas(0, 4.0, None) == dit.DIT_EINVAL
    assert dit.lib.dit_linear(7, None, 0, None, 0, 1, 1, 1, None, 0, None, None) == dit.DIT_EINVAL


def test_workspace_sizes(dit):
    cfg = dit.block_config(4096, 32, 32, 128, 12288)
    n = 4352
    ws = dit.lib.dit_block_workspace_bytes(ctypes.byref(cfg), n, 1)
    # a, o: n x 4096 bf16; qk: n x 8192 bf16; vt: 32 x 128 x n bf16; h: n x 12288 bf16
    expect = 2 * n * (4096 + 8192 + 4096 + 4096 + 12288)
    assert expect <= ws <= expect + 5 * 256
    from diffusion_transformer_image_gb300 import synth
    m = dit.model_config_from(synth.WORKLOADS["ernie_full"])
    assert dit.lib.dit_denoise_workspace_bytes(ctypes.byref(m), 64, 64, 256) > ws
    m.rope_axes[0] = 30   # axes no longer sum to head_dim
    assert dit.lib.dit_denoise_workspace_bytes(ctypes.byref(m), 64, 64, 256) == 0


def test_w8a8_workspace_and_shape_limits(dit):
    n = 4352
    bf16 = dit.block_config(4096, 32, 32, 128, 12288)
    w8 = dit.block_config(4096, 32, 32, 128, 12288, linear_format="w8a8_h256")
    ws16 = dit.lib.dit_block_workspace_bytes(ctypes.byref(bf16), n, 1)
    ws8 = dit.lib.dit_block_workspace_bytes(ctypes.byref(w8), n, 1)
    # e4m3 codes of a, o, h (1 byte each) and three row-scale vectors
    extra = n * (4096 + 4096 + 12288) + 3 * 4 * n
    assert extra <= ws8 - ws16 <= extra + 6 * 256
    # the Hadamard blocks need multiples of 256 along every contraction
    for args in ((4096 + 64, 32, 32, 128, 12288),    # hidden
                 (4096, 30, 30, 128, 12288),         # n_heads * d = 3840 is fine ...
                 (4096, 32, 32, 128, 12288 + 128)):  # ffn
        c = dit.block_config(*args, linear_format="w8a8_h256")
        ok = args[0] % 256 == 0 and (args[1] * args[3]) % 256 == 0 and args[4] % 256 == 0
        assert (dit.lib.dit_block_workspace_bytes(ctypes.byref(c), n, 1) > 0) == ok
    too_wide = dit.block_config(4096, 32, 32, 128, 16384 + 256, linear_format="w8a8_h256")
    assert dit.lib.dit_block_workspace_bytes(ctypes.byref(too_wide), n, 1) == 0
    bad_fmt = dit.block_config(4096, 32, 32, 128, 12288)
    bad_fmt.linear_format = 2
    assert dit.lib.dit_block_workspace_bytes(ctypes.byref(bad_fmt), n, 1) == 0


def test_w8a8_entry_points_reject_bad_arguments_on_host(dit):
    p = ctypes.c_void_p(4096)  # a 16-byte-aligned stand-in, never dereferenced
    s = None
    # rows not a multiple of 256 columns, or too long, or a misaligned stride
    assert dit.lib.dit_rotate_quantize(p, 300, 4, 300, p, 304, p, s) == dit.DIT_EINVAL
    assert dit.lib.dit_rotate_quantize(p, 32768, 4, 32768, p, 32768, p, s) == dit.DIT_EUNSUPPORTED
    assert dit.lib.dit_rotate_quantize(p, 1028, 4, 1024, p, 1024, p, s) == dit.DIT_EINVAL
    assert dit.lib.dit_ln_modulate_rotate_quantize(4, p, 4096, 4, 4096, p, p, 1e-6, p, 4096, p,
                                                   s) == dit.DIT_EINVAL
    assert dit.lib.dit_ln_modulate_rotate_quantize(0, p, 8448, 4, 8448, p, p, 1e-6, p, 8448, p,
                                                   s) == dit.DIT_EUNSUPPORTED
    # e4m3 linear: missing scales, K not a multiple of 16
    assert dit.lib.dit_linear_e4m3(dit.DIT_EPI_BF16, p, None, 64, p, p, 64, 4, 4, 64, p, 8, None,
                                   s) == dit.DIT_EINVAL
    assert dit.lib.dit_linear_e4m3(dit.DIT_EPI_BF16, p, p, 72, p, p, 72, 4, 4, 72, p, 8, None,
                                   s) == dit.DIT_EINVAL
    # the e4m3 QKV entry wants the W8A8 format; the bf16 one refuses it
    cfg16 = dit.block_config(4096, 32, 32, 128, 12288)
    cfg8 = dit.block_config(4096, 32, 32, 128, 12288, linear_format="w8a8_h256")
    w = dit.BlockWeights(*([4096] * len(dit.BlockWeights._fields_)))
    assert dit.lib.dit_qkv_rope_e4m3(ctypes.byref(cfg16), ctypes.byref(w), p, p, 256, 1, p, p, p,
                                     p, s) == dit.DIT_EINVAL
    assert dit.lib.dit_qkv_rope(ctypes.byref(cfg8), ctypes.byref(w), p, 256, 1, p, p, p, p,
                                s) == dit.DIT_EUNSUPPORTED
    # a W8A8 block without weight scales
    w.w_qkv_scale = None
    assert dit.lib.dit_block_forward(ctypes.byref(cfg8), ctypes.byref(w), p, 256, 1, p, p, p, p,
                                     1 << 30, s) == dit.DIT_EINVAL


def test_empty_inputs_on_host(dit):
    # zero rows: scalar arguments checked, pointers not read, nothing enqueued
    # (these return before any CUDA call, so they run without a GPU)
    L = dit.lib
    assert L.dit_ln_modulate(0, None, 1024, 0, 1024, None, None, 1e-6, None, None) == dit.DIT_OK
    assert L.dit_ln_modulate(0, None, 1024, 0, 1022, None, None, 1e-6, None, None) == dit.DIT_EINVAL
    assert L.dit_ln_modulate(0, None, 1024, -1, 1024, None, None, 1e-6, None, None) == dit.DIT_EINVAL
    assert L.dit_rotate_quantize(None, 1024, 0, 1024, None, 1024, None, None) == dit.DIT_OK
    assert L.dit_rotate_quantize(None, 1024, 0, 1000, None, 1024, None, None) == dit.DIT_EINVAL
    assert L.dit_ln_modulate_rotate_quantize(0, None, 1024, 0, 1024, None, None, 1e-6, None, 1024,
                                             None, None) == dit.DIT_OK
    assert L.flowmatch_euler_step(None, None, 0, 1.0, 0.5, None) == dit.DIT_OK
    assert L.flowmatch_euler_step(None, None, -1, 1.0, 0.5, None) == dit.DIT_EINVAL
    # an empty GEMM or token sequence is an error
    assert L.dit_linear(dit.DIT_EPI_BF16, None, 64, None, 64, 0, 64, 64, None, 64, None,
                        None) == dit.DIT_EINVAL
    cfg = dit.block_config(256, 4, 4, 64, 768)
    assert L.dit_block_workspace_bytes(ctypes.byref(cfg), 0, 1) == 0


def test_short_workspace_is_rejected_before_any_launch(dit):
    # The checks read only host values: the placeholder device addresses
    # below (16-byte aligned, never dereferenced) stand for caller buffers.
    fake = 1 << 20
    cfg = dit.block_config(256, 4, 4, 64, 768)
    w = dit.BlockWeights(*([fake] * 8))   # linears and the qk-norm gains and biases
    n = 256
    need = dit.lib.dit_block_workspace_bytes(ctypes.byref(cfg), n, 1)
    assert need > 0
    st = dit.lib.dit_block_forward(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(fake), n, 1,
                                   ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                                   ctypes.c_void_p(fake), ctypes.c_void_p(fake), need - 1, None)
    assert st == dit.DIT_EWORKSPACE
    # a misaligned workspace is an argument error, checked first
    st = dit.lib.dit_block_forward(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(fake), n, 1,
                                   ctypes.c_void_p(fake), ctypes.c_void_p(fake),
                                   ctypes.c_void_p(fake), ctypes.c_void_p(fake + 8), need, None)
    assert st == dit.DIT_EINVAL


def test_conditioning_t_dim_limit_rejected_before_any_launch(dit):
    # The time MLP's first linear stages the sinusoid in shared memory, so
    # t_dim is at most 16384: larger is DIT_EUNSUPPORTED from the host check,
    # before the weights are even looked at (they are null here, which would
    # otherwise be DIT_EINVAL) -- for the allocating and the allocation-free
    # conditioning and for the step.  t_dim = 16392 with hidden 64 stays far
    # inside the allocation-free entry point's static scratch (16392 + 128
    # floats), so this is the t_dim limit and not the scratch limit.
    from diffusion_transformer_image_gb300 import synth
    for t_dim in (16392, 16400):
        wl = synth.Workload("wide_t", hidden=64, n_heads=1, n_kv_heads=1, head_dim=64, ffn=128,
                            rope_axes=(16, 8, 8), t_dim=t_dim)
        cfg = dit.model_config_from(wl, 0)
        w = ctypes.byref(dit.ModelWeights())
        assert dit.lib.dit_timestep_conditioning_noalloc(ctypes.byref(cfg), w, 0.5, None, None,
                                                         None) == dit.DIT_EUNSUPPORTED
        assert dit.lib.dit_timestep_conditioning(ctypes.byref(cfg), w, 0.5, None, None, None,
                                                 None) == dit.DIT_EUNSUPPORTED
        assert dit.lib.dit_denoise_workspace_bytes(ctypes.byref(cfg), 8, 8, 0) == 0
    # the largest accepted t_dim passes the shape checks and stops at the null weights
    wl = synth.Workload("max_t", hidden=64, n_heads=1, n_kv_heads=1, head_dim=64, ffn=128,
                        rope_axes=(16, 8, 8), t_dim=16384)
    cfg = dit.model_config_from(wl, 0)
    assert dit.lib.dit_timestep_conditioning_noalloc(
        ctypes.byref(cfg), ctypes.byref(dit.ModelWeights()), 0.5, None, None,
        None) == dit.DIT_EINVAL
