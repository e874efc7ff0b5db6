"""The conditioning entry point that allocates nothing, for callers that may
not allocate device memory (a host that gives the library a fixed memory
budget, or a latency-critical caller for which cudaMalloc would synchronise
the device).  Its scratch is a static array inside libdit.so; its output must
match the allocating entry point's.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from diffusion_transformer_image_gb300 import synth

pytestmark = pytest.mark.gpu

dit = pytest.importorskip("diffusion_transformer_image_gb300.dit")


@pytest.mark.parametrize("name", ["tiny_block", "ernie_block"])
def test_conditioning_noalloc_matches_allocating_entry_point(name):
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda:0")
    mw = synth.model_weights(wl, seed=0, n_layers=0)
    cfg = dit.model_config_from(wl, 0)
    model = dit.DeviceModel(mw, dev, layers=[])
    H = wl.hidden
    scratch = torch.empty(wl.t_dim + 2 * H, device=dev)
    sig = dit.flowmatch_sigmas(8, 4.0)
    # two calls in a row: the second reuses the static scratch the first left
    for sigma in (sig[0], sig[5]):
        mod_ref = torch.empty(6 * H, device=dev)
        fin_ref = torch.empty(2 * H, device=dev)
        dit.dit_timestep_conditioning(cfg, model, sigma, mod_ref, fin_ref, scratch)
        mod = torch.full((6 * H,), float("nan"), device=dev)
        fin = torch.full((2 * H,), float("nan"), device=dev)
        dit.dit_timestep_conditioning_noalloc(cfg, model, sigma, mod, fin)
        torch.cuda.synchronize()
        np.testing.assert_allclose(mod.cpu().numpy(), mod_ref.cpu().numpy(), rtol=1e-6, atol=0)
        np.testing.assert_allclose(fin.cpu().numpy(), fin_ref.cpu().numpy(), rtol=1e-6, atol=0)
    assert dit.dit_last_device_error() == dit.DIT_OK


def test_conditioning_noalloc_rejects_oversize():
    # t_dim + 2 * hidden = 16400 + 16384 > 32768 floats of static scratch.
    # The size is checked on the host before anything else; the weights are
    # left null so that nothing could be launched even without that check.
    wl = synth.Workload("too_wide", hidden=8192, n_heads=64, n_kv_heads=64, head_dim=128,
                        ffn=1024, t_dim=16400)
    cfg = dit.model_config_from(wl, 0)
    st = dit.lib.dit_timestep_conditioning_noalloc(ctypes.byref(cfg), ctypes.byref(dit.ModelWeights()),
                                                   0.5, None, None, None)
    assert st == dit.DIT_EUNSUPPORTED
