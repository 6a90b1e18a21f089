// index_kernels.cu -- the block-map step: tile mean pooling, coarse scores
// with per-row top-k, and the two block indices (Q-owned and KV-owned).
//
// Pages: FastVideo test_vsa256_backward.py (_zero_pad_tail: valid tokens
// first in each tile; video_sparse_attn's topk), FastVideo
// block_sparse_attn_cute_fwd.py (_map_to_index; _build_sparse_tensors: only
// vbs > 0 tiles enter the index, and the backward index is KV-owned).
//
// Bit-exactness: pooling adds tokens in ascending order with __fadd_rn and
// divides with __fdiv_rn; scores are an __fmaf_rn chain over ascending d.
// These intrinsics are never contracted or reordered by the compiler, so
// the selection is reproducible and equals the fixed-order definition.
#include <climits>

#include "vsa_internal.h"

namespace vsa {

// ------------------------------------------------------------------ pool
// One warp per (tensor, b, h, tile); lane l owns dims 4l..4l+3 and reads 8
// bytes of each token row, so a warp reads whole 256-byte rows (coalesced),
// 16 rows in flight, and adds them in ascending token order. The tensors of
// one call (q and k, or q, k and v) share one launch, so small problems
// still fill the GPU.
template <typename T>
__global__ void __launch_bounds__(256) k_pool(Prob p, PoolSegs segs) {
    long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    int si = 0;
    while (si < segs.n && w >= segs.s[si].warps) {
        w -= segs.s[si].warps;
        ++si;
    }
    if (si >= segs.n) return;
    const bool q_side = segs.s[si].q_side != 0;
    const T *x = static_cast<const T *>(segs.s[si].x);
    float *out = segs.s[si].out;
    const int H = q_side ? p.Hq : p.Hkv, nT = q_side ? p.nQ : p.nKV;
    const int Tt = q_side ? p.tile_q : p.tile_kv;
    const int t = (int)(w % nT), h = (int)((w / nT) % H), b = (int)(w / ((long long)nT * H));
    const int lane = threadIdx.x & 31;
    const int var = q_side ? q_valid(p, b, t) : kv_valid(p, b, t);
    const long long rs = (p.layout == L_BHSD) ? p.D : (long long)H * p.D;  // token stride
    const T *base = x + tok_off(p, q_side, b, t * Tt, h) + lane * 4;
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    int r = 0;
    for (; r + 16 <= var; r += 16) {
        uint2 buf[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) buf[u] = __ldg(reinterpret_cast<const uint2 *>(base + (long long)(r + u) * rs));
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            float2 a = unpack2<T>(buf[u].x), c = unpack2<T>(buf[u].y);
            s[0] = __fadd_rn(s[0], a.x);
            s[1] = __fadd_rn(s[1], a.y);
            s[2] = __fadd_rn(s[2], c.x);
            s[3] = __fadd_rn(s[3], c.y);
        }
    }
    for (; r < var; ++r) {
        uint2 v = __ldg(reinterpret_cast<const uint2 *>(base + (long long)r * rs));
        float2 a = unpack2<T>(v.x), c = unpack2<T>(v.y);
        s[0] = __fadd_rn(s[0], a.x);
        s[1] = __fadd_rn(s[1], a.y);
        s[2] = __fadd_rn(s[2], c.x);
        s[3] = __fadd_rn(s[3], c.y);
    }
    float4 o;
    const float fv = (float)var;
    o.x = var > 0 ? __fdiv_rn(s[0], fv) : 0.f;
    o.y = var > 0 ? __fdiv_rn(s[1], fv) : 0.f;
    o.z = var > 0 ? __fdiv_rn(s[2], fv) : 0.f;
    o.w = var > 0 ? __fdiv_rn(s[3], fv) : 0.f;
    *reinterpret_cast<float4 *>(out + w * p.D + lane * 4) = o;
}

cudaError_t launch_pools(const Prob &p, const PoolSegs &segs_in, cudaStream_t s) {
    PoolSegs segs = segs_in;
    long long warps = 0;
    for (int i = 0; i < segs.n; ++i) {
        const bool q = segs.s[i].q_side != 0;
        segs.s[i].warps = (long long)p.B * (q ? p.Hq : p.Hkv) * (q ? p.nQ : p.nKV);
        warps += segs.s[i].warps;
    }
    const long long blocks = (warps + 7) / 8;
    if (blocks == 0) return cudaSuccess;
    prof_begin("pool", s);
    if (p.dtype == T_BF16)
        k_pool<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(p, segs);
    else
        k_pool<__half><<<(unsigned)blocks, 256, 0, s>>>(p, segs);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_pool_qkv(const Prob &p, const void *q, float *pq, const void *k, float *pk, const void *v,
                            float *pv, cudaStream_t s) {
    // a tensor given as NULL is not pooled (its means are kept from an earlier call)
    PoolSegs segs{};
    if (q) segs.s[segs.n++] = PoolSeg{q, pq, 1, 0};
    if (k) segs.s[segs.n++] = PoolSeg{k, pk, 0, 0};
    if (v) segs.s[segs.n++] = PoolSeg{v, pv, 0, 0};
    if (segs.n == 0) return cudaSuccess;
    return launch_pools(p, segs, s);
}

// ---------------------------------------------------------------- select
// Block = 8 warps = 8 * RPW query tiles of one (b, h); warp w owns query
// tiles i0 + w * RPW .. + RPW - 1. Key-tile means are staged through shared
// memory in chunks of 128 tiles with 16-byte copies (rows padded to 132
// floats, so the 16-byte reads of eight lanes at a time hit distinct bank
// groups). Lane l computes the scores of tiles l, l+32, l+64, l+96 of a
// chunk for the warp's RPW query tiles; every score is one __fmaf_rn chain
// over ascending d, as in the fixed-order definition.
//
// Top-k: scores map to order-preserving 32-bit keys (-0 folded into +0, so
// equal scores give equal keys); a radix search over four 8-bit digits
// (a 256-bin histogram per warp and pass) finds the k-th largest key T
// (the largest T with at least k keys >= T). The selection is every key > T
// plus the lowest-indexed keys == T up to k, which is the repeated-argmax
// rule with ties to the lower tile index.
constexpr int kSelChunk = 128;
constexpr int kSelPitch = 132;

__device__ __forceinline__ uint32_t score_key(float x) {
    if (x == 0.f) x = 0.f;
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int RPW>
__global__ void __launch_bounds__(256) k_select(Prob p, const float *__restrict__ pq,
                                                const float *__restrict__ pk, int topk, uint8_t *map,
                                                int *q_idx, int *q_cnt, int cap) {
    constexpr int R = 8 * RPW;
    extern __shared__ __align__(16) float sm[];
    float *spk = sm;                                  // [kSelChunk][kSelPitch]
    float *spq = spk + kSelChunk * kSelPitch;         // [R][128]
    float *ssc = spq + R * 128;                       // [R][nKV]
    int *shist = reinterpret_cast<int *>(ssc + R * p.nKV) + (threadIdx.x >> 5) * 256;  // this warp's 256 bins
    const int b = blockIdx.z, h = blockIdx.y, hk = h / (p.Hq / p.Hkv);
    const int i0 = blockIdx.x * R, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = 128;
    for (int e = threadIdx.x; e < R * D / 4; e += blockDim.x) {
        const int r = e / (D / 4), ii = i0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ii < p.nQ) v = __ldg(reinterpret_cast<const float4 *>(pq + (((long long)b * p.Hq + h) * p.nQ + ii) * D) + (e % (D / 4)));
        reinterpret_cast<float4 *>(spq)[e] = v;
    }
    const float *pkh = pk + ((long long)b * p.Hkv + hk) * p.nKV * D;
    // The next chunk of key means is loaded into registers while the current
    // one is scored, and stored to shared memory at the top of the next pass.
    float4 buf[16];
    auto load_chunk = [&](int j0) {
        const int nj = min(kSelChunk, p.nKV - j0);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int e = threadIdx.x + u * 256;  // 4096 16-byte words per full chunk
            buf[u] = e < nj * (D / 4) ? __ldg(reinterpret_cast<const float4 *>(pkh + (long long)j0 * D) + e)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    load_chunk(0);
    for (int j0 = 0; j0 < p.nKV; j0 += kSelChunk) {
        const int nj = min(kSelChunk, p.nKV - j0);
        __syncthreads();  // the previous chunk is scored
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int e = threadIdx.x + u * 256;
            if (e < nj * (D / 4))
                *reinterpret_cast<float4 *>(spk + (e / (D / 4)) * kSelPitch + (e % (D / 4)) * 4) = buf[u];
        }
        __syncthreads();
        if (j0 + kSelChunk < p.nKV) load_chunk(j0 + kSelChunk);
        float acc[RPW][4];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[r][u] = 0.f;
        const float *aq = spq + (w * RPW) * D;
#pragma unroll 2
        for (int e = 0; e < D; e += 4) {
            float4 c4[4], a4[RPW];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                c4[u] = *reinterpret_cast<const float4 *>(spk + (lane + 32 * u) * kSelPitch + e);
#pragma unroll
            for (int r = 0; r < RPW; ++r) a4[r] = *reinterpret_cast<const float4 *>(aq + r * D + e);
#pragma unroll
            for (int r = 0; r < RPW; ++r)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc[r][u] = __fmaf_rn(a4[r].x, c4[u].x, acc[r][u]);
                    acc[r][u] = __fmaf_rn(a4[r].y, c4[u].y, acc[r][u]);
                    acc[r][u] = __fmaf_rn(a4[r].z, c4[u].z, acc[r][u]);
                    acc[r][u] = __fmaf_rn(a4[r].w, c4[u].w, acc[r][u]);
                }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int jj = lane + 32 * u;
            if (jj < nj) {
                const bool valid = kv_valid(p, b, j0 + jj) > 0;
#pragma unroll
                for (int r = 0; r < RPW; ++r) ssc[(w * RPW + r) * p.nKV + j0 + jj] = valid ? acc[r][u] : -INFINITY;
            }
        }
    }
    __syncwarp();
    for (int r = 0; r < RPW; ++r) {
        const int i = i0 + w * RPW + r;
        if (i >= p.nQ) break;
        const long long row = ((long long)b * p.Hq + h) * p.nQ + i;
        const float *sc = ssc + (w * RPW + r) * p.nKV;
        const int k = q_rows(p, b, i) > 0 ? min(topk, p.nKV) : 0;
        uint32_t T = 0xFFFFFFFFu;  // no key reaches it: nothing selected when k = 0
        int need = 0;             // keys == T to take, lowest index first
        if (k > 0) {
            // T is found 8 bits at a time from the top: among the keys that
            // match the bits found so far, the digit at which the count of
            // keys with a larger digit first reaches `rem` (the keys still
            // to take); those larger keys are taken and leave `rem`. After
            // the last digit, rem = the keys == T to take.
            uint32_t prefix = 0u, known = 0u;
            int rem = k;
#pragma unroll 1
            for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u) shist[lane * 8 + u] = 0;
                __syncwarp();
                for (int j = lane; j < p.nKV; j += 32) {
                    const uint32_t key = score_key(sc[j]);
                    if ((key & known) == prefix) atomicAdd(&shist[(key >> shift) & 255u], 1);
                }
                __syncwarp();
                // lane l holds the digits 255 - 8l down to 248 - 8l
                int c[8], sum = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    c[u] = shist[255 - 8 * lane - u];
                    sum += c[u];
                }
                int inc = sum;  // keys with digits from 255 down to this lane's last
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, inc, off);
                    if (lane >= off) inc += y;
                }
                const int exc = inc - sum;
                const int L = __ffs(__ballot_sync(0xffffffffu, exc < rem && inc >= rem)) - 1;
                int digit = 0, above = 0;
                if (lane == L) {
                    int acc = exc;
                    bool found = false;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {  // the first digit (descending) whose count reaches rem
                        const bool here = !found && acc + c[u] >= rem;
                        digit = here ? 255 - 8 * lane - u : digit;
                        above = here ? acc : above;
                        found = found || here;
                        acc += c[u];
                    }
                }
                digit = __shfl_sync(0xffffffffu, digit, L);
                above = __shfl_sync(0xffffffffu, above, L);
                rem -= above;
                prefix |= (uint32_t)digit << shift;
                known |= 255u << shift;
                __syncwarp();  // every lane has read the bins before the next pass clears them
            }
            T = prefix;
            need = rem;
        }
        int cnt = 0, taken = 0;
        for (int j0 = 0; j0 < p.nKV; j0 += 32) {
            const int j = j0 + lane;
            const bool inb = k > 0 && j < p.nKV;
            const uint32_t key = inb ? score_key(sc[j]) : 0u;
            const bool tie = inb && key == T;
            const unsigned eq = __ballot_sync(0xffffffffu, tie);
            const bool on = inb && (key > T || (tie && taken + __popc(eq & ((1u << lane) - 1u)) < need));
            taken += __popc(eq);
            if (j < p.nKV) map[row * p.nKV + j] = on ? 1 : 0;
            const bool f = on && kv_valid(p, b, j) > 0;
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            if (f) q_idx[row * cap + cnt + __popc(bal & ((1u << lane) - 1u))] = j;
            cnt += __popc(bal);
        }
        for (int n = cnt + lane; n < cap; n += 32) q_idx[row * cap + n] = -1;
        if (lane == 0) q_cnt[row] = cnt;
    }
}

size_t select_smem(int rpw, int nKV) {
    return sizeof(float) * ((size_t)kSelChunk * kSelPitch + (size_t)8 * rpw * 128 + (size_t)8 * rpw * nKV) +
           sizeof(int) * 8 * 256;  // one 256-bin histogram per warp
}

cudaError_t launch_select(const Prob &p, const float *pq, const float *pk, int topk, uint8_t *map, int *q_idx,
                          int *q_cnt, int cap, cudaStream_t s) {
    const size_t cap_smem = 227 * 1024;
    // two query tiles per warp: two blocks fit on an SM for the usual tile counts
    const int rpw = select_smem(2, p.nKV) <= cap_smem ? 2 : 1;
    const cudaError_t ae = rpw == 2 ? ensure_smem_limit((const void *)k_select<2>, (int)cap_smem)
                                    : ensure_smem_limit((const void *)k_select<1>, (int)cap_smem);
    if (ae != cudaSuccess) return ae;
    const int R = 8 * rpw;
    dim3 grid((p.nQ + R - 1) / R, p.Hq, p.B);
    prof_begin("select_topk", s);
    if (rpw == 2)
        k_select<2><<<grid, 256, select_smem(2, p.nKV), s>>>(p, pq, pk, topk, map, q_idx, q_cnt, cap);
    else
        k_select<1><<<grid, 256, select_smem(1, p.nKV), s>>>(p, pq, pk, topk, map, q_idx, q_cnt, cap);
    prof_end(s);
    return cudaGetLastError();
}

// ------------------------------------------------------------ mask index
// One warp per (b, h, query tile): ballot-compact the marked tiles that
// hold valid tokens, ascending.
__global__ void __launch_bounds__(256) k_mask_index(Prob p, const uint8_t *__restrict__ map, int *q_idx,
                                                    int *q_cnt, int cap) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= (long long)p.B * p.Hq * p.nQ) return;
    const int lane = threadIdx.x & 31;
    const int i = (int)(row % p.nQ), b = (int)(row / ((long long)p.nQ * p.Hq));
    const bool exists = q_rows(p, b, i) > 0;
    int cnt = 0;
    for (int j0 = 0; j0 < p.nKV; j0 += 32) {
        const int j = j0 + lane;
        const bool f = exists && j < p.nKV && map[row * p.nKV + j] != 0 && kv_valid(p, b, j) > 0;
        const unsigned bal = __ballot_sync(0xffffffffu, f);
        if (f) q_idx[row * cap + cnt + __popc(bal & ((1u << lane) - 1u))] = j;
        cnt += __popc(bal);
    }
    for (int n = cnt + lane; n < cap; n += 32) q_idx[row * cap + n] = -1;
    if (lane == 0) q_cnt[row] = cnt;
}

cudaError_t launch_mask_index(const Prob &p, const uint8_t *map, int *q_idx, int *q_cnt, int cap,
                              cudaStream_t s) {
    const long long rows = (long long)p.B * p.Hq * p.nQ;
    if (rows == 0) return cudaSuccess;
    prof_begin("mask_index", s);
    k_mask_index<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, map, q_idx, q_cnt, cap);
    prof_end(s);
    return cudaGetLastError();
}

// ------------------------------------------------------------- transpose
// One block per (b, h). Thread-per-KV-tile column scans of the map count
// the selecting query tiles, a block-wide exclusive scan gives kv_ptr, and
// a second column scan writes the lists in ascending query-tile order. An
// entry counts iff the map marks it, the KV tile holds valid tokens and the
// query tile exists -- the same filter that built the Q-owned index.
__global__ void __launch_bounds__(1024) k_transpose(Prob p, const uint8_t *__restrict__ map, int *kv_ptr,
                                                    int *kv_qidx, int cap) {
    extern __shared__ int cnt[];  // [nKV + 1]
    __shared__ int warp_tot[32];
    const int b = blockIdx.y, h = blockIdx.x;
    const long long bh = (long long)b * p.Hq + h;
    const uint8_t *m = map + bh * p.nQ * p.nKV;
    for (int j = threadIdx.x; j < p.nKV; j += blockDim.x) {
        int c = 0;
        if (kv_valid(p, b, j) > 0)
            for (int i = 0; i < p.nQ; ++i) c += (m[(long long)i * p.nKV + j] != 0 && q_rows(p, b, i) > 0);
        cnt[j] = c;
    }
    __syncthreads();
    // exclusive scan of cnt[0..nKV) into cnt[0..nKV], thread t owns a segment
    const int per = (p.nKV + blockDim.x - 1) / blockDim.x;
    const int lo = min(p.nKV, (int)threadIdx.x * per), hi = min(p.nKV, lo + per);
    int local = 0;
    for (int j = lo; j < hi; ++j) local += cnt[j];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += y;
        }
        warp_tot[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    int run = (incl - local) + (wid > 0 ? warp_tot[wid - 1] : 0);
    int *ptr = kv_ptr + bh * (p.nKV + 1);
    for (int j = lo; j < hi; ++j) {
        const int c = cnt[j];
        ptr[j] = run;
        run += c;
    }
    const int total = warp_tot[(blockDim.x >> 5) - 1];
    if (threadIdx.x == 0) ptr[p.nKV] = total;
    __syncthreads();
    int *lst = kv_qidx + bh * (long long)p.nQ * cap;
    for (int j = threadIdx.x; j < p.nKV; j += blockDim.x) {
        int pos = ptr[j];
        if (kv_valid(p, b, j) > 0)
            for (int i = 0; i < p.nQ; ++i)
                if (m[(long long)i * p.nKV + j] != 0 && q_rows(p, b, i) > 0) lst[pos++] = i;
    }
    for (long long n = total + threadIdx.x; n < (long long)p.nQ * cap; n += blockDim.x) lst[n] = -1;
}

cudaError_t launch_transpose(const Prob &p, const uint8_t *map, int *kv_ptr, int *kv_qidx, int cap,
                             cudaStream_t s) {
    if (p.B == 0 || p.Hq == 0) return cudaSuccess;
    dim3 grid(p.Hq, p.B);
    const size_t smem = sizeof(int) * (p.nKV + 1);
    const cudaError_t ae = ensure_smem_limit((const void *)k_transpose, 64 * 1024);
    if (ae != cudaSuccess) return ae;
    prof_begin("transpose_index", s);
    k_transpose<<<grid, 1024, smem, s>>>(p, map, kv_ptr, kv_qidx, cap);
    prof_end(s);
    return cudaGetLastError();
}

// ------------------------------------------------------------ query blocks
// A caller's mask at query-block granularity: block_q rows (dividing
// tile_q) x one KV tile, [B, Hq, nQb, nKV] ([NPU-test]: block_shape
// [32, 128] and [64, 128]). The attention kernels keep tiles of tile_q
// rows: a tile attends to the union of its blocks' selections, and a bit
// mask per (tile, selected KV tile) -- bit s set iff block s of the tile
// selected it -- masks the keys row by row.
namespace {

__device__ __forceinline__ bool block_exists(const Prob &p, int b, int i, int s, int bq, int nQb) {
    const int blk = i * (p.tile_q / bq) + s;
    if (blk >= nQb) return false;
    if (p.layout == L_TND) return i * p.tile_q + s * bq < seq_len(p, true, b);
    return true;
}
__device__ __forceinline__ int tile_bits(const Prob &p, const uint8_t *__restrict__ bm, int nQb, int bq, int b,
                                         int h, int i, int j) {
    const int ns = p.tile_q / bq;
    const uint8_t *m = bm + ((long long)b * p.Hq + h) * nQb * p.nKV;
    int bits = 0;
    for (int sb = 0; sb < ns; ++sb)
        if (block_exists(p, b, i, sb, bq, nQb) && m[(long long)(i * ns + sb) * p.nKV + j] != 0) bits |= 1 << sb;
    return bits;
}

// tile map = union over each tile's blocks
__global__ void __launch_bounds__(256) k_block_union(Prob p, int bq, int nQb, const uint8_t *__restrict__ bm,
                                                     uint8_t *__restrict__ tmap) {
    const long long n = (long long)p.B * p.Hq * p.nQ * p.nKV;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n;
         x += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(x % p.nKV);
        const long long r = x / p.nKV;
        const int i = (int)(r % p.nQ), h = (int)((r / p.nQ) % p.Hq), b = (int)(r / ((long long)p.nQ * p.Hq));
        tmap[x] = tile_bits(p, bm, nQb, bq, b, h, i, j) != 0;
    }
}

// bit masks of the Q-owned index entries and, when kv_ptr is given, of the
// KV-owned ones (entry pos of KV tile j: kv_ptr[j] <= pos < kv_ptr[j+1])
__global__ void __launch_bounds__(256) k_block_bits(Prob p, int bq, int nQb, const uint8_t *__restrict__ bm,
                                                    const int *__restrict__ q_idx, const int *__restrict__ q_cnt,
                                                    int cap, int *__restrict__ q_sub, const int *__restrict__ kv_ptr,
                                                    const int *__restrict__ kv_qidx, int *__restrict__ kv_qsub) {
    const long long n = (long long)p.B * p.Hq * p.nQ * cap;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n;
         x += (long long)gridDim.x * blockDim.x) {
        const long long r = x / cap;  // (b, h, i) row of the Q-owned index; also the KV-owned list's entry
        const int slot = (int)(x % cap);
        const int i = (int)(r % p.nQ), h = (int)((r / p.nQ) % p.Hq), b = (int)(r / ((long long)p.nQ * p.Hq));
        q_sub[x] = slot < q_cnt[r] ? tile_bits(p, bm, nQb, bq, b, h, i, q_idx[x]) : 0;
        if (kv_ptr) {
            // entry pos of head (b, h)'s KV-owned list
            const long long bh = (long long)b * p.Hq + h;
            const long long pos = x - bh * p.nQ * cap;
            const int *ptr = kv_ptr + bh * (p.nKV + 1);
            int bits = 0;
            if (pos < ptr[p.nKV]) {
                int lo = 0, hi = p.nKV;  // largest j with ptr[j] <= pos
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (ptr[mid] <= pos) lo = mid; else hi = mid;
                }
                bits = tile_bits(p, bm, nQb, bq, b, h, kv_qidx[bh * p.nQ * cap + pos], lo);
            }
            kv_qsub[x] = bits;
        }
    }
}

int grid_for(long long n) {
    const long long g = (n + 255) / 256;
    return (int)(g < 1 ? 1 : (g > 65535 ? 65535 : g));
}

}  // namespace

cudaError_t launch_block_index(const Prob &p, int bq, int nQb, const uint8_t *bm, uint8_t *tmap, int *q_idx,
                               int *q_cnt, int *q_sub, int cap, int *kv_ptr, int *kv_qidx, int *kv_qsub,
                               cudaStream_t s) {
    prof_begin("block_union", s);
    k_block_union<<<grid_for((long long)p.B * p.Hq * p.nQ * p.nKV), 256, 0, s>>>(p, bq, nQb, bm, tmap);
    prof_end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if ((e = launch_mask_index(p, tmap, q_idx, q_cnt, cap, s)) != cudaSuccess) return e;
    if (kv_ptr && (e = launch_transpose(p, tmap, kv_ptr, kv_qidx, cap, s)) != cudaSuccess) return e;
    prof_begin("block_bits", s);
    k_block_bits<<<grid_for((long long)p.B * p.Hq * p.nQ * cap), 256, 0, s>>>(p, bq, nQb, bm, q_idx, q_cnt, cap, q_sub,
                                                                            kv_ptr, kv_qidx, kv_qsub);
    prof_end(s);
    return cudaGetLastError();
}

}  // namespace vsa
