"""GB300 diffusion-transformer hot path: Python binding of libdit.so.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  Importing
this package fails loudly when libdit.so has not been built; there is no
other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))  # the package directory
LIB_PATH = os.path.join(_PKG, "libdit.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first "
        "(python -m diffusion_transformer_image_gb300.build)")

lib = ctypes.CDLL(LIB_PATH)

c_int32, c_int64, c_float, c_size_t, c_void_p = (
    ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p)
c_float_p = ctypes.POINTER(ctypes.c_float)

DIT_OK, DIT_EINVAL, DIT_EUNSUPPORTED, DIT_EWORKSPACE, DIT_ECUDA, DIT_ETIMEOUT = 0, -1, -2, -3, -4, -5
DIT_EPI_BF16, DIT_EPI_F32_BIAS, DIT_EPI_RESIDUAL, DIT_EPI_SWIGLU = 0, 1, 2, 3
DIT_EPI_GEGLU, DIT_EPI_RESIDUAL_TANH, DIT_EPI_RESIDUAL_SIGMOID = 4, 5, 6
NORM_KINDS = {"layer": 0, "rms": 1}
GLU_ACTS = {"silu": 0, "gelu_tanh": 1}
ROPE_ORDERS = {"norm_rope": 0, "rope_norm": 1}
GATE_FNS = {"identity": 0, "tanh": 1, "sigmoid": 2}
LINEAR_FORMATS = {"bf16": 0, "w8a8_h256": 1}

EXPORTED = [
    "dit_block_workspace_bytes", "dit_block_forward", "dit_denoise_workspace_bytes",
    "dit_denoise_step", "flowmatch_euler_step", "flowmatch_sigmas", "dit_linear",
    "dit_qkv_rope", "dit_qkv_rope_e4m3", "dit_attention", "dit_ln_modulate",
    "dit_rotate_quantize", "dit_ln_modulate_rotate_quantize", "dit_linear_e4m3",
    "dit_timestep_conditioning",
    "dit_timestep_conditioning_noalloc",
    "dit_rope_table_grid", "dit_rope_table_pos", "dit_rope_table_vit",
    "dit_last_device_error", "dit_set_wait_timeout_ns", "dit_debug_stuck_wait",
    "dit_launch_count", "dit_status_string",
]


class DitError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {lib.dit_status_string(status).decode()} ({status})")
        self.status = status


class BlockConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("n_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("ffn", c_int32), ("rope_layout", c_int32),
                ("adaln", c_int32), ("qk_norm", c_int32), ("ln_eps", c_float),
                ("norm_kind", c_int32), ("glu_act", c_int32), ("rope_order", c_int32),
                ("gate_fn", c_int32), ("linear_format", c_int32)]


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("w_qkv", "w_o", "w_gu", "w_down", "q_g", "q_b", "k_g",
                                        "k_b", "ln1_g", "ln1_b", "ln2_g", "ln2_b",
                                        "w_qkv_scale", "w_o_scale", "w_gu_scale",
                                        "w_down_scale")]


class ModelConfig(ctypes.Structure):
    _fields_ = [("block", BlockConfig), ("n_layers", c_int32), ("latent_channels", c_int32),
                ("t_dim", c_int32), ("t_scale", c_float), ("rope_axes", c_int32 * 3),
                ("rope_theta", c_float)]


class ModelWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("patch_w", "patch_b", "t_w1", "t_b1", "t_w2", "t_b2",
                                        "mod_w", "mod_b", "fin_w", "fin_b", "out_w", "out_b")]
    _fields_ += [("layers", ctypes.POINTER(BlockWeights))]


def _sig(name, res, args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = args
    return f


_P = ctypes.POINTER
_sig("dit_status_string", ctypes.c_char_p, [c_int32])
_sig("dit_block_workspace_bytes", c_size_t, [_P(BlockConfig), c_int32, c_int32])
_sig("dit_block_forward", c_int32, [_P(BlockConfig), _P(BlockWeights), c_void_p, c_int32, c_int32,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p])
_sig("dit_denoise_workspace_bytes", c_size_t, [_P(ModelConfig), c_int32, c_int32, c_int32])
_sig("dit_denoise_step", c_int32, [_P(ModelConfig), _P(ModelWeights), c_void_p, c_void_p, c_int32,
                                   c_int32, c_int32, c_float, c_float, c_void_p, c_void_p,
                                   c_size_t, c_void_p])
_sig("flowmatch_euler_step", c_int32, [c_void_p, c_void_p, c_int64, c_float, c_float, c_void_p])
_sig("flowmatch_sigmas", c_int32, [c_int32, c_float, c_float_p])
_sig("dit_linear", c_int32, [c_int32, c_void_p, c_int64, c_void_p, c_int64, c_int32, c_int32,
                             c_int32, c_void_p, c_int64, c_void_p, c_void_p])
_sig("dit_qkv_rope", c_int32, [_P(BlockConfig), _P(BlockWeights), c_void_p, c_int32, c_int32,
                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p])
_sig("dit_qkv_rope_e4m3", c_int32, [_P(BlockConfig), _P(BlockWeights), c_void_p, c_void_p,
                                    c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p])
_sig("dit_attention", c_int32, [_P(BlockConfig), c_void_p, c_void_p, c_int32, c_int32, c_void_p,
                                c_void_p])
_sig("dit_ln_modulate", c_int32, [c_int32, c_void_p, c_int64, c_int32, c_int32, c_void_p, c_void_p,
                                  c_float, c_void_p, c_void_p])
_sig("dit_rotate_quantize", c_int32, [c_void_p, c_int64, c_int32, c_int32, c_void_p, c_int64,
                                      c_void_p, c_void_p])
_sig("dit_ln_modulate_rotate_quantize", c_int32, [c_int32, c_void_p, c_int64, c_int32, c_int32,
                                                  c_void_p, c_void_p, c_float, c_void_p, c_int64,
                                                  c_void_p, c_void_p])
_sig("dit_linear_e4m3", c_int32, [c_int32, c_void_p, c_void_p, c_int64, c_void_p, c_void_p,
                                  c_int64, c_int32, c_int32, c_int32, c_void_p, c_int64, c_void_p,
                                  c_void_p])
_sig("dit_timestep_conditioning", c_int32, [_P(ModelConfig), _P(ModelWeights), c_float, c_void_p,
                                            c_void_p, c_void_p, c_void_p])
_sig("dit_timestep_conditioning_noalloc", c_int32, [_P(ModelConfig), _P(ModelWeights), c_float,
                                                    c_void_p, c_void_p, c_void_p])
_sig("dit_rope_table_grid", c_int32, [c_int32, c_int32, c_int32, _P(c_int32), c_float, c_void_p,
                                      c_void_p, c_void_p])
_sig("dit_rope_table_pos", c_int32, [c_void_p, c_int32, _P(c_int32), c_float, c_void_p, c_void_p,
                                     c_void_p])
_sig("dit_rope_table_vit", c_int32, [c_int32, c_int32, c_int32, c_int32, c_float, c_void_p,
                                     c_void_p, c_void_p])
_sig("dit_last_device_error", c_int32, [c_void_p])
_sig("dit_set_wait_timeout_ns", c_int32, [ctypes.c_uint64])
_sig("dit_debug_stuck_wait", c_int32, [c_void_p])
_sig("dit_launch_count", c_int64, [c_int32])


def _check(status: int, where: str):
    if status != DIT_OK:
        raise DitError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# --------------------------------------------------------------- structures
def block_config(hidden, n_heads, n_kv_heads, head_dim, ffn, rope_layout="interleaved",
                 adaln=True, qk_norm=True, ln_eps=1e-6, norm_kind="layer", glu="silu",
                 rope_order="norm_rope", gate_fn="identity",
                 linear_format="bf16") -> BlockConfig:
    return BlockConfig(hidden, n_heads, n_kv_heads, head_dim, ffn,
                       0 if rope_layout == "interleaved" else 1, int(bool(adaln)),
                       int(bool(qk_norm)), ln_eps, NORM_KINDS[norm_kind], GLU_ACTS[glu],
                       ROPE_ORDERS[rope_order], GATE_FNS[gate_fn],
                       LINEAR_FORMATS[linear_format])


def block_config_from(wl) -> BlockConfig:
    """BlockConfig of a synthetic workload description (synth.Workload)."""
    return block_config(wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.ffn,
                        wl.rope_layout, wl.adaln, wl.qk_norm, norm_kind=wl.norm_kind,
                        glu=wl.glu, rope_order=wl.rope_order, gate_fn=wl.gate_fn,
                        linear_format=wl.linear_format)


def model_config_from(wl, n_layers: Optional[int] = None) -> ModelConfig:
    m = ModelConfig()
    m.block = block_config_from(wl)
    m.n_layers = wl.n_layers if n_layers is None else n_layers
    m.latent_channels = wl.latent_channels
    m.t_dim = wl.t_dim
    m.t_scale = 1000.0
    m.rope_axes = (c_int32 * 3)(*wl.rope_axes)
    m.rope_theta = wl.rope_theta
    return m


LINEAR_KEYS = ("w_qkv", "w_o", "w_gu", "w_down")


class DeviceBlock:
    """One block's weights resident on the GPU, with the C structure that
    points at them (the tensors are kept alive by this object).  With
    linear_format "w8a8_h256" the four projection weights are rotated and
    coded on the GPU (dit_rotate_quantize) and only the codes and their row
    scales are kept."""

    def __init__(self, w: dict, device="cuda", linear_format: str = "bf16"):
        def dev(t, dtype):
            return None if t is None else t.to(device=device, dtype=dtype).contiguous()
        self.t = {k: dev(w.get(k), torch.bfloat16) for k in LINEAR_KEYS}
        for k in ("q_g", "q_b", "k_g", "k_b", "ln1_g", "ln1_b", "ln2_g", "ln2_b"):
            self.t[k] = dev(w.get(k), torch.float32)
        for k in LINEAR_KEYS:
            self.t[k + "_scale"] = None
        if LINEAR_FORMATS[linear_format] == LINEAR_FORMATS["w8a8_h256"]:
            for k in LINEAR_KEYS:
                self.t[k], self.t[k + "_scale"] = dit_rotate_quantize(self.t[k])
        self.c = BlockWeights(*[(None if self.t[n] is None else self.t[n].data_ptr())
                                for n, _ in BlockWeights._fields_])


class DeviceModel:
    """Denoiser weights resident on the GPU."""

    def __init__(self, mw: dict, device="cuda", layers=None, linear_format: str = "bf16"):
        self.t = {}
        for k in ("patch_w", "t_w1", "t_w2", "mod_w", "fin_w", "out_w"):
            self.t[k] = mw[k].to(device=device, dtype=torch.bfloat16).contiguous()
        for k in ("patch_b", "t_b1", "t_b2", "mod_b", "fin_b", "out_b"):
            self.t[k] = mw[k].to(device=device, dtype=torch.float32).contiguous()
        self.blocks = layers if layers is not None else [
            DeviceBlock(l, device, linear_format) for l in mw["layers"]]
        self.layer_array = (BlockWeights * max(1, len(self.blocks)))(*[b.c for b in self.blocks])
        self.c = ModelWeights(*[self.t[n].data_ptr() for n, _ in ModelWeights._fields_[:-1]])
        self.c.layers = ctypes.cast(self.layer_array, ctypes.POINTER(BlockWeights))


# --------------------------------------------------------------- the path
def dit_block_workspace_bytes(cfg: BlockConfig, n_tokens: int, n_seqs: int = 1) -> int:
    return lib.dit_block_workspace_bytes(ctypes.byref(cfg), n_tokens, n_seqs)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def dit_block_forward(cfg: BlockConfig, w: DeviceBlock, x: torch.Tensor, mod, rope_cos,
                      rope_sin, n_seqs: int = 1, ws: Optional[torch.Tensor] = None, stream=None):
    n = x.shape[0]
    if ws is None:
        ws = workspace(dit_block_workspace_bytes(cfg, n, n_seqs), x.device)
    _check(lib.dit_block_forward(ctypes.byref(cfg), None if w is None else ctypes.byref(w.c),
                                 _ptr(x), n, n_seqs,
                                 _ptr(mod), _ptr(rope_cos), _ptr(rope_sin), _ptr(ws),
                                 ws.numel(), _stream(stream)), "dit_block_forward")
    return x


def dit_denoise_workspace_bytes(cfg: ModelConfig, grid_h: int, grid_w: int, n_txt: int) -> int:
    return lib.dit_denoise_workspace_bytes(ctypes.byref(cfg), grid_h, grid_w, n_txt)


def dit_denoise_step(cfg: ModelConfig, w: DeviceModel, latent: torch.Tensor, text, grid_h: int,
                     grid_w: int, sigma: float, sigma_next: float, velocity_out=None,
                     ws: Optional[torch.Tensor] = None, stream=None):
    n_txt = 0 if text is None else text.shape[0]
    if ws is None:
        ws = workspace(dit_denoise_workspace_bytes(cfg, grid_h, grid_w, n_txt), latent.device)
    _check(lib.dit_denoise_step(ctypes.byref(cfg), ctypes.byref(w.c), _ptr(latent), _ptr(text),
                                grid_h, grid_w, n_txt, sigma, sigma_next, _ptr(velocity_out),
                                _ptr(ws), ws.numel(), _stream(stream)), "dit_denoise_step")
    return latent


def flowmatch_euler_step(x: torch.Tensor, v: torch.Tensor, sigma: float, sigma_next: float,
                         stream=None):
    _check(lib.flowmatch_euler_step(_ptr(x), _ptr(v), x.numel(), sigma, sigma_next,
                                    _stream(stream)), "flowmatch_euler_step")
    return x


def flowmatch_sigmas(n_steps: int, shift: float) -> list:
    buf = (c_float * (n_steps + 1))()
    _check(lib.flowmatch_sigmas(n_steps, shift, buf), "flowmatch_sigmas")
    return list(buf)


def dit_linear(epilogue: int, a: torch.Tensor, w: torch.Tensor, out: torch.Tensor,
               bias_or_gate=None, n_out: Optional[int] = None, stream=None):
    M, K = a.shape
    glu = epilogue in (DIT_EPI_SWIGLU, DIT_EPI_GEGLU)
    N = n_out if n_out is not None else (w.shape[0] // 2 if glu else w.shape[0])
    _check(lib.dit_linear(epilogue, _ptr(a), a.stride(0), _ptr(w), w.stride(0), M, N, K, _ptr(out),
                          out.stride(0), _ptr(bias_or_gate), _stream(stream)), "dit_linear")
    return out


def dit_qkv_rope(cfg: BlockConfig, w: DeviceBlock, a, rope_cos, rope_sin, qk, vt, n_seqs=1,
                 stream=None):
    _check(lib.dit_qkv_rope(ctypes.byref(cfg), ctypes.byref(w.c), _ptr(a), a.shape[0], n_seqs,
                            _ptr(rope_cos), _ptr(rope_sin), _ptr(qk), _ptr(vt), _stream(stream)),
           "dit_qkv_rope")


def dit_qkv_rope_e4m3(cfg: BlockConfig, w: DeviceBlock, a, a_scales, rope_cos, rope_sin, qk, vt,
                      n_seqs=1, stream=None):
    _check(lib.dit_qkv_rope_e4m3(ctypes.byref(cfg), ctypes.byref(w.c), _ptr(a), _ptr(a_scales),
                                 a.shape[0], n_seqs, _ptr(rope_cos), _ptr(rope_sin), _ptr(qk),
                                 _ptr(vt), _stream(stream)), "dit_qkv_rope_e4m3")


def dit_attention(cfg: BlockConfig, qk, vt, o, n_seqs=1, stream=None):
    """qk: [n_heads + n_kv_heads, n_tokens, d] bf16 (head-major); vt as written
    by dit_qkv_rope; o: [n_tokens, n_heads * d] bf16."""
    _check(lib.dit_attention(ctypes.byref(cfg), _ptr(qk), _ptr(vt), o.shape[0], n_seqs, _ptr(o),
                             _stream(stream)), "dit_attention")
    return o


def dit_ln_modulate(mode: int, x: torch.Tensor, p0, p1, eps: float, out: torch.Tensor,
                    stream=None):
    rows, H = x.shape
    _check(lib.dit_ln_modulate(mode, _ptr(x), x.stride(0), rows, H, _ptr(p0), _ptr(p1), eps,
                               _ptr(out), _stream(stream)), "dit_ln_modulate")
    return out


def dit_rotate_quantize(x: torch.Tensor, codes: Optional[torch.Tensor] = None,
                        scales: Optional[torch.Tensor] = None, stream=None):
    """Rows of bf16 x [rows, K] rotated by the 256-point Hadamard matrix and
    coded in e4m3: returns (codes uint8 [rows, K], scales fp32 [rows])."""
    rows, K = x.shape
    if codes is None:
        codes = torch.empty(rows, K, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(lib.dit_rotate_quantize(_ptr(x), x.stride(0), rows, K, _ptr(codes), codes.stride(0),
                                   _ptr(scales), _stream(stream)), "dit_rotate_quantize")
    return codes, scales


def dit_ln_modulate_rotate_quantize(mode: int, x: torch.Tensor, p0, p1, eps: float,
                                    codes: torch.Tensor, scales: torch.Tensor, stream=None):
    rows, H = x.shape
    _check(lib.dit_ln_modulate_rotate_quantize(mode, _ptr(x), x.stride(0), rows, H, _ptr(p0),
                                               _ptr(p1), eps, _ptr(codes), codes.stride(0),
                                               _ptr(scales), _stream(stream)),
           "dit_ln_modulate_rotate_quantize")
    return codes, scales


def dit_linear_e4m3(epilogue: int, a: torch.Tensor, a_scales: torch.Tensor, w: torch.Tensor,
                    w_scales: torch.Tensor, out: torch.Tensor, bias_or_gate=None,
                    n_out: Optional[int] = None, stream=None):
    """dit_linear on e4m3 codes (uint8 tensors) with per-row scales."""
    M, K = a.shape
    glu = epilogue in (DIT_EPI_SWIGLU, DIT_EPI_GEGLU)
    N = n_out if n_out is not None else (w.shape[0] // 2 if glu else w.shape[0])
    _check(lib.dit_linear_e4m3(epilogue, _ptr(a), _ptr(a_scales), a.stride(0), _ptr(w),
                               _ptr(w_scales), w.stride(0), M, N, K, _ptr(out), out.stride(0),
                               _ptr(bias_or_gate), _stream(stream)), "dit_linear_e4m3")
    return out


def dit_timestep_conditioning(cfg: ModelConfig, w: DeviceModel, sigma: float, mod, fin, scratch,
                              stream=None):
    _check(lib.dit_timestep_conditioning(ctypes.byref(cfg), ctypes.byref(w.c), sigma, _ptr(mod),
                                         _ptr(fin), _ptr(scratch), _stream(stream)),
           "dit_timestep_conditioning")


def dit_timestep_conditioning_noalloc(cfg: ModelConfig, w: DeviceModel, sigma: float, mod, fin,
                                      stream=None):
    """dit_timestep_conditioning without a scratch argument: for callers that
    may not allocate device memory (the scratch is a static array in the
    library).  Calls that overlap on the GPU race on that array."""
    _check(lib.dit_timestep_conditioning_noalloc(ctypes.byref(cfg), ctypes.byref(w.c), sigma,
                                                 _ptr(mod), _ptr(fin), _stream(stream)),
           "dit_timestep_conditioning_noalloc")


def dit_rope_table_grid(grid_h: int, grid_w: int, n_txt: int, axes: Sequence[int], theta: float,
                        cos_out, sin_out, stream=None):
    """cos_out, sin_out: device fp32 [d/2, grid_h*grid_w + n_txt] (pair-major)."""
    ax = (c_int32 * 3)(*axes)
    _check(lib.dit_rope_table_grid(grid_h, grid_w, n_txt, ax, theta, _ptr(cos_out), _ptr(sin_out),
                                   _stream(stream)), "dit_rope_table_grid")


def dit_rope_table_pos(pos: torch.Tensor, axes: Sequence[int], theta: float, cos_out, sin_out,
                       stream=None):
    """cos_out, sin_out: device fp32 [d/2, n] (pair-major) for pos [n, 3]."""
    ax = (c_int32 * 3)(*axes)
    _check(lib.dit_rope_table_pos(_ptr(pos), pos.shape[0], ax, theta, _ptr(cos_out), _ptr(sin_out),
                                  _stream(stream)), "dit_rope_table_pos")


def dit_rope_table_vit(grid_h: int, grid_w: int, n_prefix: int, head_dim: int, base: float,
                       cos_out, sin_out, stream=None):
    """cos_out, sin_out: device fp32 [head_dim/2, n_prefix + grid_h*grid_w]."""
    _check(lib.dit_rope_table_vit(grid_h, grid_w, n_prefix, head_dim, base, _ptr(cos_out),
                                  _ptr(sin_out), _stream(stream)), "dit_rope_table_vit")


def dit_last_device_error(stream=None) -> int:
    return lib.dit_last_device_error(_stream(stream))


def dit_set_wait_timeout_ns(ns: int):
    _check(lib.dit_set_wait_timeout_ns(ns), "dit_set_wait_timeout_ns")


def dit_debug_stuck_wait(stream=None):
    _check(lib.dit_debug_stuck_wait(_stream(stream)), "dit_debug_stuck_wait")


def dit_launch_count(reset: bool = False) -> int:
    return lib.dit_launch_count(1 if reset else 0)
