// vsa_common.cuh -- problem description, indexing and small device helpers
// shared by the library's kernels. Internal to libvsa.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vsa {

enum { L_BHSD = 0, L_BSHD = 1, L_TND = 2 };
enum { T_BF16 = 0, T_FP16 = 1 };

// Problem description passed to kernels by value.
struct Prob {
    int layout, dtype;
    int B, Hq, Hkv, D;
    int Sq, Skv;          // padded per-batch tokens, or totals in TND
    int tile_q, tile_kv;
    int nQ, nKV;
    const int *cu_q, *cu_kv;     // TND offsets (device)
    const int *q_var, *kv_var;   // padded-layout tile fills (device)
    float scale;
};

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// TND: first token and length of sequence b, with the offsets clamped into
// [0, total tokens] (a decreasing or overlong offset array cannot move an
// access outside the tensor; vsa_check_inputs reports such arrays).
__device__ __forceinline__ int seq_start(const Prob &p, bool q_side, int b) {
    return clampi((q_side ? p.cu_q : p.cu_kv)[b], 0, q_side ? p.Sq : p.Skv);
}
__device__ __forceinline__ int seq_len(const Prob &p, bool q_side, int b) {
    const int s0 = seq_start(p, q_side, b);
    return clampi((q_side ? p.cu_q : p.cu_kv)[b + 1], s0, q_side ? p.Sq : p.Skv) - s0;
}

// Valid tokens of KV tile j of batch entry b (padded layouts: kv_var[j]
// clamped to [0, tile]; a value outside that range is invalid input, which
// vsa_check_inputs reports; TND: the part of the tile inside the sequence).
__device__ __forceinline__ int kv_valid(const Prob &p, int b, int j) {
    if (p.layout == L_TND) return clampi(seq_len(p, false, b) - j * p.tile_kv, 0, p.tile_kv);
    return clampi(p.kv_var[j], 0, p.tile_kv);
}
__device__ __forceinline__ int q_valid(const Prob &p, int b, int i) {
    if (p.layout == L_TND) return clampi(seq_len(p, true, b) - i * p.tile_q, 0, p.tile_q);
    return clampi(p.q_var[i], 0, p.tile_q);
}
// Query rows of tile i that exist (all slots in the padded layouts).
__device__ __forceinline__ int q_rows(const Prob &p, int b, int i) {
    return p.layout == L_TND ? q_valid(p, b, i) : p.tile_q;
}
// Element offset of (batch b, token s within b, head h, d = 0).
__device__ __forceinline__ long long tok_off(const Prob &p, bool q_side, int b, int s, int h) {
    const int H = q_side ? p.Hq : p.Hkv;
    if (p.layout == L_BHSD) {
        const int S = q_side ? p.Sq : p.Skv;
        return (((long long)b * H + h) * S + s) * p.D;
    }
    if (p.layout == L_BSHD) {
        const int S = q_side ? p.Sq : p.Skv;
        return (((long long)b * S + s) * H + h) * p.D;
    }
    return ((long long)(seq_start(p, q_side, b) + s) * H + h) * p.D;
}
// Offset of the LSE / Dvec entry of (b, h, s): [B, Hq, Sq] or [Hq, T].
__device__ __forceinline__ long long lse_off(const Prob &p, int b, int h, int s) {
    if (p.layout == L_TND) return (long long)h * p.Sq + seq_start(p, true, b) + s;
    return ((long long)b * p.Hq + h) * p.Sq + s;
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// Two floats packed to one 32-bit word of 16-bit values (lo = a).
template <typename T> __device__ __forceinline__ uint32_t pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w));
}
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<__half2 *>(&w));
}

// The 128-key chunks of a query tile's selected KV tiles, walked by a whole
// warp: a window of up to 32 selected tiles sits one tile per lane (tile
// id, valid key count, chunk count and first chunk within the window), so
// the index is read once per 32 tiles rather than once per chunk, and a
// chunk's tile is found with a ballot. All lanes call with the same c.
struct ChunkWin {
    const int *idx, *sub;  // sub: query-block bit masks of the entries (NULL: whole tiles)
    int cnt, per;
    int n0, c0, chunks;  // first tile and first chunk of the window; chunks in it
    int j, kvv, nch, first, bits;  // this lane's tile
};
__device__ __forceinline__ void win_load(const Prob &p, int b, ChunkWin &w, int lane) {
    const int n = w.n0 + lane;
    w.j = n < w.cnt ? w.idx[n] : 0;
    // tile ids outside [0, nKV) (invalid input) contribute no chunk
    w.kvv = (n < w.cnt && w.j >= 0 && w.j < p.nKV) ? kv_valid(p, b, w.j) : 0;
    w.bits = (n < w.cnt && w.sub) ? w.sub[n] : -1;
    w.nch = min(w.per, (w.kvv + 127) >> 7);
    int inc = w.nch;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    w.first = inc - w.nch;
    w.chunks = __shfl_sync(0xffffffffu, inc, 31);
}
__device__ __forceinline__ ChunkWin win_begin(const Prob &p, int b, const int *idx, const int *sub, int cnt,
                                               int lane) {
    ChunkWin w;
    w.idx = idx;
    w.sub = sub;
    w.cnt = cnt;  // already clamped into [0, idx_cap] by the caller
    w.per = p.tile_kv >> 7;
    w.n0 = 0;
    w.c0 = 0;
    win_load(p, b, w, lane);
    return w;
}
// Row (of the KV tile's first key, within the batch entry) and valid key
// count of chunk c; chunks are visited in increasing order.
__device__ __forceinline__ bool win_chunk(const Prob &p, int b, ChunkWin &w, int c, int lane, int &row, int &valid,
                                          int &bits) {
    while (c >= w.c0 + w.chunks) {
        if (w.n0 + 32 >= w.cnt) return false;
        w.c0 += w.chunks;
        w.n0 += 32;
        win_load(p, b, w, lane);
    }
    const int cw = c - w.c0;
    const unsigned m = __ballot_sync(0xffffffffu, w.nch > 0 && w.first <= cw);
    const int L = 31 - __clz(m);
    const int first = __shfl_sync(0xffffffffu, w.first, L);
    const int kvv = __shfl_sync(0xffffffffu, w.kvv, L);
    const int j = __shfl_sync(0xffffffffu, w.j, L);
    bits = __shfl_sync(0xffffffffu, w.bits, L);
    const int sub = cw - first;
    row = j * p.tile_kv + sub * 128;
    valid = min(128, kvv - sub * 128);
    return true;
}

// Device status word (first bytes of the caller's workspace).
__device__ __forceinline__ void set_error(unsigned *err, unsigned code) {
    if (err) atomicCAS(err, 0u, code);
}

}  // namespace vsa
