// tile3d.cu -- the layout step on either side of the attention: scatter a
// video latent [B, T, H, W, R] (R = heads x head_dim elements per token)
// into padded 3D tiles [B, nTiles * tile, R] and gather it back.
//
// Pages: FastVideo test_vsa256_backward.py (_BLOCK_SIZE_3D = (4, 8, 8) with
// product 256; _zero_pad_tail: callers scatter into a zeroed tile buffer, so
// the first var slots of a tile are its tokens and the rest are zero). The
// order of tiles and of tokens inside a tile is not on the pages; here both
// are raster order (tiles over (T, H, W) tile coordinates; the tokens of a
// tile over its own, possibly clipped, (t, h, w) box), so a tile's valid
// count is the product of its clipped extents.
//
// Both directions move whole token rows (R elements, contiguous in both
// layouts): one warp per destination row, 16-byte vector copies, several
// rows per warp in flight across the grid. HBM-bound: 2 x B x nTokens x R
// bytes moved (plus the zero padding written by tile_3d).
#include <cstdint>

#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

struct Tiling {
    int B, T, H, W;          // latent grid
    int tT, tH, tW;          // tile box
    int nT, nH, nW;          // tiles along each axis (ceil)
    int tile;                // tT * tH * tW slots per tile
    long long row16;         // 16-byte words per token row
};

__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }

// Source token (within batch entry) of slot `s` of tile `k`, or -1 for a
// padding slot.
__device__ __forceinline__ long long slot_source(const Tiling &g, int k, int s) {
    const int wi = k % g.nW, hi = (k / g.nW) % g.nH, ti = k / (g.nW * g.nH);
    const int et = imin(g.tT, g.T - ti * g.tT), eh = imin(g.tH, g.H - hi * g.tH), ew = imin(g.tW, g.W - wi * g.tW);
    if (s >= et * eh * ew) return -1;
    const int lw = s % ew, lh = (s / ew) % eh, lt = s / (ew * eh);
    return ((long long)(ti * g.tT + lt) * g.H + (hi * g.tH + lh)) * g.W + (wi * g.tW + lw);
}

// latent -> tiles (padding slots written as zeros); also the per-tile valid
// counts when `tile_var` is given.
__global__ void __launch_bounds__(256) k_tile_3d(Tiling g, const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                 int32_t *__restrict__ tile_var) {
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int ntiles = g.nT * g.nH * g.nW;
    const long long rows = (long long)g.B * ntiles * g.tile;
    const long long ntok = (long long)g.T * g.H * g.W;
    if (tile_var) {
        const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
        if (t < ntiles) {
            const int k = (int)t;
            const int wi = k % g.nW, hi = (k / g.nW) % g.nH, ti = k / (g.nW * g.nH);
            tile_var[k] = imin(g.tT, g.T - ti * g.tT) * imin(g.tH, g.H - hi * g.tH) * imin(g.tW, g.W - wi * g.tW);
        }
    }
    for (long long row = warp0; row < rows; row += nwarps) {
        const int b = (int)(row / ((long long)ntiles * g.tile));
        const int rem = (int)(row - (long long)b * ntiles * g.tile);
        const long long s = slot_source(g, rem / g.tile, rem % g.tile);
        uint4 *d = dst + row * g.row16;
        if (s < 0) {
            for (long long u = lane; u < g.row16; u += 32) d[u] = make_uint4(0, 0, 0, 0);
        } else {
            const uint4 *p = src + ((long long)b * ntok + s) * g.row16;
            for (long long u = lane; u < g.row16; u += 32) d[u] = __ldg(p + u);
        }
    }
}

// tiles -> latent (padding slots are not read).
__global__ void __launch_bounds__(256) k_untile_3d(Tiling g, const uint4 *__restrict__ src, uint4 *__restrict__ dst) {
    const int lane = threadIdx.x & 31;
    const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int ntiles = g.nT * g.nH * g.nW;
    const long long ntok = (long long)g.T * g.H * g.W;
    const long long rows = (long long)g.B * ntok;
    for (long long row = warp0; row < rows; row += nwarps) {
        const int b = (int)(row / ntok);
        const long long tok = row - (long long)b * ntok;
        const int w = (int)(tok % g.W), h = (int)((tok / g.W) % g.H), t = (int)(tok / ((long long)g.W * g.H));
        const int ti = t / g.tT, hi = h / g.tH, wi = w / g.tW;
        const int lt = t - ti * g.tT, lh = h - hi * g.tH, lw = w - wi * g.tW;
        const int eh = imin(g.tH, g.H - hi * g.tH), ew = imin(g.tW, g.W - wi * g.tW);
        const int k = (ti * g.nH + hi) * g.nW + wi;
        const int slot = (lt * eh + lh) * ew + lw;
        const uint4 *p = src + ((long long)b * ntiles * g.tile + (long long)k * g.tile + slot) * g.row16;
        uint4 *d = dst + row * g.row16;
        for (long long u = lane; u < g.row16; u += 32) d[u] = __ldg(p + u);
    }
}

vsa_status make_tiling(int B, int T, int H, int W, int row_bytes, int tT, int tH, int tW, Tiling *g) {
    if (B < 1 || T < 1 || H < 1 || W < 1 || tT < 1 || tH < 1 || tW < 1) return VSA_ERR_SHAPE;
    if (row_bytes < 16 || row_bytes % 16 != 0) return VSA_ERR_SHAPE;
    g->B = B; g->T = T; g->H = H; g->W = W;
    g->tT = tT; g->tH = tH; g->tW = tW;
    g->nT = (T + tT - 1) / tT; g->nH = (H + tH - 1) / tH; g->nW = (W + tW - 1) / tW;
    const long long tile = (long long)tT * tH * tW;
    const long long ntiles = (long long)g->nT * g->nH * g->nW;
    if (tile > (1 << 20) || ntiles * tile > (1LL << 31) - 1 || (long long)T * H * W > (1LL << 31) - 1)
        return VSA_ERR_UNSUPPORTED;
    g->tile = (int)tile;
    g->row16 = row_bytes / 16;
    return VSA_OK;
}

int tiling_grid(long long rows) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (rows + 7) / 8;  // 8 warps (rows) per block
    const long long cap = (long long)sms * 8;  // 8 blocks of 256 threads per SM
    return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" int vsa_tile_3d_count(int T, int H, int W, int tT, int tH, int tW) {
    if (T < 1 || H < 1 || W < 1 || tT < 1 || tH < 1 || tW < 1) return -1;
    return ((T + tT - 1) / tT) * ((H + tH - 1) / tH) * ((W + tW - 1) / tW);
}

extern "C" vsa_status vsa_tile_3d(int B, int T, int H, int W, int row_bytes, int tT, int tH, int tW,
                                  const void *latent, void *tiled, int32_t *tile_var, vsa_stream_t stream) {
    if (!latent || !tiled) return VSA_ERR_NULL;
    if (((uintptr_t)latent | (uintptr_t)tiled) & 15u) return VSA_ERR_LAYOUT;
    Tiling g;
    const vsa_status st = make_tiling(B, T, H, W, row_bytes, tT, tH, tW, &g);
    if (st != VSA_OK) return st;
    const long long rows = (long long)B * g.nT * g.nH * g.nW * g.tile;
    const long long ntiles = (long long)g.nT * g.nH * g.nW;
    long long grid = tiling_grid(rows);
    if (tile_var && grid * 256 < ntiles) grid = (ntiles + 255) / 256;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    prof_begin("tile_3d", s);
    k_tile_3d<<<(int)grid, 256, 0, s>>>(g, static_cast<const uint4 *>(latent), static_cast<uint4 *>(tiled), tile_var);
    prof_end(s);
    return status_from_cuda(cudaGetLastError());
}

extern "C" vsa_status vsa_untile_3d(int B, int T, int H, int W, int row_bytes, int tT, int tH, int tW,
                                    const void *tiled, void *latent, vsa_stream_t stream) {
    if (!latent || !tiled) return VSA_ERR_NULL;
    if (((uintptr_t)latent | (uintptr_t)tiled) & 15u) return VSA_ERR_LAYOUT;
    Tiling g;
    const vsa_status st = make_tiling(B, T, H, W, row_bytes, tT, tH, tW, &g);
    if (st != VSA_OK) return st;
    const long long rows = (long long)B * T * H * W;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    prof_begin("untile_3d", s);
    k_untile_3d<<<tiling_grid(rows), 256, 0, s>>>(g, static_cast<const uint4 *>(tiled), static_cast<uint4 *>(latent));
    prof_end(s);
    return status_from_cuda(cudaGetLastError());
}
