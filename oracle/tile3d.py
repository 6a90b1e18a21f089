"""Oracle of the 3D video tiling (numpy, plain loops over tiles).

TEST INFRASTRUCTURE. Only tests/ and the benchmark import this module.

FastVideo test_vsa256_backward.py fixes the tile box (_BLOCK_SIZE_3D =
(4, 8, 8), 256 slots) and that a tile's tokens occupy its first var slots
with the rest zero (_zero_pad_tail: callers scatter into a zeroed tile
buffer). The orders are not on the page; the reading taken here is raster
order for the tiles over their (T, H, W) tile coordinates and raster order
for the tokens of a tile over its own box clipped at the latent's edges.
"""
from __future__ import annotations

import numpy as np


def tile_count(T: int, H: int, W: int, tile=(4, 8, 8)) -> int:
    tT, tH, tW = tile
    return (-(-T // tT)) * (-(-H // tH)) * (-(-W // tW))


def tile_3d(latent: np.ndarray, tile=(4, 8, 8)):
    """latent [B, T, H, W, ...] -> (tiled [B, nTiles * prod(tile), ...],
    tile_var [nTiles] int32)."""
    B, T, H, W = latent.shape[:4]
    rest = latent.shape[4:]
    tT, tH, tW = tile
    nT, nH, nW = -(-T // tT), -(-H // tH), -(-W // tW)
    slots = tT * tH * tW
    tiled = np.zeros((B, nT * nH * nW * slots) + rest, dtype=latent.dtype)
    tile_var = np.zeros(nT * nH * nW, dtype=np.int32)
    k = 0
    for ti in range(nT):
        for hi in range(nH):
            for wi in range(nW):
                box = latent[:, ti * tT:(ti + 1) * tT, hi * tH:(hi + 1) * tH, wi * tW:(wi + 1) * tW]
                n = box.shape[1] * box.shape[2] * box.shape[3]
                tiled[:, k * slots:k * slots + n] = box.reshape((B, n) + rest)
                tile_var[k] = n
                k += 1
    return tiled, tile_var


def untile_3d(tiled: np.ndarray, grid, tile=(4, 8, 8)) -> np.ndarray:
    """tiled [B, nTiles * prod(tile), ...] -> latent [B, T, H, W, ...]."""
    T, H, W = grid
    B = tiled.shape[0]
    rest = tiled.shape[2:]
    tT, tH, tW = tile
    nT, nH, nW = -(-T // tT), -(-H // tH), -(-W // tW)
    slots = tT * tH * tW
    latent = np.zeros((B, T, H, W) + rest, dtype=tiled.dtype)
    k = 0
    for ti in range(nT):
        for hi in range(nH):
            for wi in range(nW):
                t0, h0, w0 = ti * tT, hi * tH, wi * tW
                et, eh, ew = min(tT, T - t0), min(tH, H - h0), min(tW, W - w0)
                n = et * eh * ew
                latent[:, t0:t0 + et, h0:h0 + eh, w0:w0 + ew] = \
                    tiled[:, k * slots:k * slots + n].reshape((B, et, eh, ew) + rest)
                k += 1
    return latent
