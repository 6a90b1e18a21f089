"""GPU parity of the 3D video tiling kernels (vsa_tile_3d / vsa_untile_3d)
against the oracle's per-tile loops: bit-exact (pure data movement)."""
import numpy as np
import pytest
import torch

from oracle import tile3d as otile
from bwd_tile_mean_gb300 import vsa

pytestmark = pytest.mark.gpu

CASES = [
    # (B, (T, H, W), trailing row shape, dtype, tile box)
    (1, (4, 8, 8), (2, 128), torch.bfloat16, (4, 8, 8)),
    (2, (5, 9, 7), (3, 128), torch.float16, (4, 8, 8)),
    (1, (21, 45, 80), (1, 8), torch.bfloat16, (4, 8, 8)),   # the gated-ragged KV grid, 16-byte rows
    (3, (6, 17, 3), (4, 64), torch.bfloat16, (2, 4, 4)),
    (1, (1, 1, 1), (1, 128), torch.float16, (4, 8, 8)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-{c[1][0]}x{c[1][1]}x{c[1][2]}-{c[4][0]}{c[4][1]}{c[4][2]}")
def test_tile_untile_bit_exact(case):
    B, grid, rest, dtype, box = case
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn((B,) + grid + rest, generator=g, device="cuda", dtype=torch.float32).to(dtype)
    tiled, var = vsa.tile_3d(x, box)
    ref_tiled, ref_var = otile.tile_3d(x.cpu().view(torch.int16).numpy(), box)
    np.testing.assert_array_equal(tiled.cpu().view(torch.int16).numpy(), ref_tiled)
    np.testing.assert_array_equal(var.cpu().numpy(), ref_var)
    back = vsa.untile_3d(tiled, grid, box)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    torch.cuda.synchronize()


def test_video_dit_latent_full_size():
    """The 76,800-token latent (20x48x80, 40 heads x 128, bf16; 786 MB):
    the box divides the grid, so tiling equals the reshape/transpose block
    permutation; untiling restores the latent bit for bit."""
    T, H, W, heads, D = 20, 48, 80, 40, 128
    g = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randn((1, T, H, W, heads, D), generator=g, device="cuda", dtype=torch.bfloat16)
    tiled, var = vsa.tile_3d(x, (4, 8, 8))
    assert tiled.shape == (1, 76800, heads, D) and var.shape == (300,)
    assert bool((var == 256).all())
    ref = x.view(1, T // 4, 4, H // 8, 8, W // 8, 8, heads, D).permute(0, 1, 3, 5, 2, 4, 6, 7, 8)
    assert torch.equal(tiled.view(torch.int16), ref.reshape(1, 76800, heads, D).view(torch.int16))
    back = vsa.untile_3d(tiled, (T, H, W), (4, 8, 8))
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    del x, tiled, back, ref
    torch.cuda.empty_cache()


def test_host_validation():
    x = torch.zeros((1, 4, 8, 8, 1, 4), device="cuda", dtype=torch.bfloat16)  # 8-byte rows
    with pytest.raises(vsa.VsaError):
        vsa.tile_3d(x, (4, 8, 8))
