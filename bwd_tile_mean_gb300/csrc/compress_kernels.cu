// compress_kernels.cu -- the gated compression branch, forward and backward.
//
// Pages: FastVideo test_vsa256_backward.py
// (test_vsa256_cute_backward_with_compress_gate: out = sparse_out + gate *
// compress_out, the gate without a gradient). Per query tile i of head h,
// with the fp32 tile means pq (query tiles) and pk, pv (key/value tiles,
// head h / (Hq / Hkv)):
//   a_ij = scale pq_i . pk_j over the key/value tiles with valid tokens,
//   A_i  = softmax_j(a_ij),  c_i = sum_j A_ij pv_j;
// backward, with dc_i = sum over the tile's query rows of gate (*) dO:
//   dA_ij = dc_i . pv_j,  ds_ij = A_ij (dA_ij - sum_j A_ij dA_ij),
//   dpq_i = scale sum_j ds_ij pk_j,
//   dpk_j = scale sum_{h, i} ds_ij pq_i,  dpv_j = sum_{h, i} A_ij dc_i
// (the last two summed over the GQA group's query heads).
//
// These are small fp32 products ([nQ x 128] by [128 x nKV] per head), so
// the kernels are bound by how often they read the pooled means, not by
// arithmetic. A CTA takes up to kCQ query tiles of one head and streams
// the head's key/value means through shared memory in chunks of kCJ tiles
// (rows padded to kCPitch floats, so the lanes of a warp, which read
// different tiles at the same dimension, hit distinct banks): each mean is
// read from L2 once per kCQ query tiles instead of once per query tile.
// The column pass takes kCJB key/value tiles per CTA and streams the query
// side. Sums run in a fixed order, so every result is the same on every run.
#include "vsa_internal.h"

namespace vsa {
namespace {

constexpr int kCQ = 16;        // query tiles per CTA (row passes), at most
constexpr int kCJ = 32;        // key/value tiles per staged chunk
constexpr int kCPitch = 132;   // floats per staged row (16-byte aligned; 8 lanes' 16-byte reads hit distinct banks)
constexpr int kCJB = 16;       // key/value tiles per CTA (column pass)
constexpr int kCThreads = 256;

// Floats per row of the [query tile][key/value tile] score and A / ds
// rows held in shared memory: nKV rounded up to a multiple of 4, so that
// four consecutive tiles' values are one 16-byte read.
__host__ __device__ __forceinline__ int nkv_pitch(const Prob &p) { return (p.nKV + 3) & ~3; }
__device__ __forceinline__ float4 ld4(const float *x) { return *reinterpret_cast<const float4 *>(x); }
// a (+)= x . y over 4 consecutive dims, in dim order
__device__ __forceinline__ float dot4(float4 x, float4 y, float a) {
    a = fmaf(x.x, y.x, a);
    a = fmaf(x.y, y.y, a);
    a = fmaf(x.z, y.z, a);
    return fmaf(x.w, y.w, a);
}
// acc[u] += sum over jj of sS[(q0 + u) pitch + j0 + jj] st[jj][d], jj in
// ascending order (rows q0 + u < nq); four jj per 16-byte read of sS.
__device__ __forceinline__ void acc_staged(float (&acc)[8], const float *sS, int pitch, int j0, int nj,
                                           const float *st, int d, int q0, int nq) {
    int jj = 0;
    for (; jj + 4 <= nj; jj += 4) {
        const float v0 = st[jj * kCPitch + d], v1 = st[(jj + 1) * kCPitch + d];
        const float v2 = st[(jj + 2) * kCPitch + d], v3 = st[(jj + 3) * kCPitch + d];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (q0 + u < nq) {
                const float4 a = ld4(sS + (q0 + u) * pitch + j0 + jj);
                acc[u] = fmaf(a.x, v0, acc[u]);
                acc[u] = fmaf(a.y, v1, acc[u]);
                acc[u] = fmaf(a.z, v2, acc[u]);
                acc[u] = fmaf(a.w, v3, acc[u]);
            }
    }
    for (; jj < nj; ++jj) {
        const float v = st[jj * kCPitch + d];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (q0 + u < nq) acc[u] = fmaf(sS[(q0 + u) * pitch + j0 + jj], v, acc[u]);
    }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Rows [j0, j0 + nj) of a [nKV, 128] fp32 matrix, staged through shared
// memory as st[kCJ][kCPitch] in two steps: chunk_load issues a thread's
// four 16-byte loads into registers, chunk_store writes them. The passes
// below load chunk n + 1 right after storing chunk n, so its L2 round trip
// overlaps the arithmetic on chunk n.
static_assert(kCJ * 32 == 4 * kCThreads, "a chunk is four 16-byte loads per thread");
__device__ __forceinline__ int chunk_rows(int nKV, int j0) { return j0 < nKV ? min(kCJ, nKV - j0) : 0; }
__device__ __forceinline__ void chunk_load(float4 (&v)[4], const float *__restrict__ src, int j0, int nj) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src + (long long)j0 * 128);
    const int n4 = nj * 32;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int x = threadIdx.x + k * kCThreads;
        v[k] = x < n4 ? s4[x] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
__device__ __forceinline__ void chunk_store(float *st, const float4 (&v)[4], int nj) {
    const int n4 = nj * 32;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int x = threadIdx.x + k * kCThreads;
        if (x < n4) *reinterpret_cast<float4 *>(st + (x >> 5) * kCPitch + (x & 31) * 4) = v[k];
    }
}
// Copy n floats (a multiple of 4; both sides 16-byte aligned) into shared
// memory, eight 16-byte loads in flight per thread.
__device__ __forceinline__ void load_rows(float *dst, const float *__restrict__ src, int n) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int x0 = 0; x0 < n / 4; x0 += 8 * kCThreads) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int x = x0 + threadIdx.x + k * kCThreads;
            if (x < n / 4) v[k] = s4[x];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int x = x0 + threadIdx.x + k * kCThreads;
            if (x < n / 4) d4[x] = v[k];
        }
    }
}

// Row r of sA: the softmax of its nKV scores in place (-inf: no valid
// token; a row with none stays all zero). One warp.
__device__ __forceinline__ void softmax_row(float *r, int n, int lane) {
    float mx = -INFINITY;
    for (int j = lane; j < n; j += 32) mx = fmaxf(mx, r[j]);
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j < n; j += 32) {
        const float e = r[j] == -INFINITY ? 0.f : __expf(r[j] - mx);
        r[j] = e;
        sum += e;
    }
    sum = warp_sum(sum);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int j = lane; j < n; j += 32) r[j] *= inv;
}

// ------------------------------------------------------------- forward
// CTA (b, h, query tiles [i0, i0 + qb)): scores against every key/value
// tile, row softmax, c = A pv.
__global__ void __launch_bounds__(kCThreads) k_compress_fwd(Prob p, const float *__restrict__ pq,
                                                          const float *__restrict__ pk,
                                                          const float *__restrict__ pv, float *__restrict__ c,
                                                          int qb) {
    extern __shared__ __align__(16) float sm[];
    float *sq = sm;                      // [kCQ][128] this CTA's query means
    float *st = sq + kCQ * 128;          // [kCJ][kCPitch] staged pk, then pv
    float *sA = st + kCJ * kCPitch;      // [qb][nkv_pitch] scores, then A
    const int h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    const int pa = nkv_pitch(p);
    const int i0 = blockIdx.x * qb, nq = min(qb, p.nQ - i0);
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const long long row0 = ((long long)b * p.Hq + h) * p.nQ + i0;
    const float *pkh = pk + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    const float *pvh = pv + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    float4 pf[4];
    chunk_load(pf, pkh, 0, chunk_rows(p.nKV, 0));
    load_rows(sq, pq + row0 * 128, nq * 128);
    // scores: thread (tile j0 + lane, rows w and w + 8; a row past nq is
    // computed from whatever sq holds there and not stored)
    for (int j0 = 0; j0 < p.nKV; j0 += kCJ) {
        const int nj = min(kCJ, p.nKV - j0);
        __syncthreads();
        chunk_store(st, pf, nj);
        __syncthreads();
        if (j0 + kCJ < p.nKV) chunk_load(pf, pkh, j0 + kCJ, chunk_rows(p.nKV, j0 + kCJ));
        else chunk_load(pf, pvh, 0, chunk_rows(p.nKV, 0));  // the c pass's first chunk
        if (lane < nj && w < nq) {
            const bool valid = kv_valid(p, b, j0 + lane) > 0;
            const int w2 = min(w + 8, kCQ - 1);
            float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
            for (int d = 0; d < 128; d += 4) {
                const float4 kd = ld4(st + lane * kCPitch + d);
                a0 = dot4(ld4(sq + w * 128 + d), kd, a0);
                a1 = dot4(ld4(sq + w2 * 128 + d), kd, a1);
            }
            sA[w * pa + j0 + lane] = valid ? a0 * p.scale : -INFINITY;
            if (w + 8 < nq) sA[(w + 8) * pa + j0 + lane] = valid ? a1 * p.scale : -INFINITY;
        }
    }
    __syncthreads();
    for (int q = w; q < nq; q += 8) softmax_row(sA + q * pa, p.nKV, lane);
    // c = A pv: thread (dim t % 128, rows 8 (t / 128) .. + 8)
    const int d = t & 127, q0 = (t >> 7) * 8;
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int j0 = 0; j0 < p.nKV; j0 += kCJ) {
        const int nj = min(kCJ, p.nKV - j0);
        __syncthreads();
        chunk_store(st, pf, nj);
        __syncthreads();
        if (j0 + kCJ < p.nKV) chunk_load(pf, pvh, j0 + kCJ, chunk_rows(p.nKV, j0 + kCJ));
        acc_staged(acc, sA, pa, j0, nj, st, d, q0, nq);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (q0 + u < nq) c[(row0 + q0 + u) * 128 + d] = acc[u];
}

// ------------------------------------------------------------ backward
// dc_i = sum over the query rows of tile i of gate (*) dO (fp32, per dim).
// Thread: 8 dims (one 16-byte load of each tensor), rows phase, phase + 8,
// ..., four rows' loads issued before their sums (taken in row order); the
// eight phases' partial sums are added in a fixed order.
template <typename T>
__global__ void __launch_bounds__(128) k_compress_dc(Prob p, const T *__restrict__ dO, const T *__restrict__ gate,
                                                     float *__restrict__ dc) {
    __shared__ float part[8][128];
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, e0 = (t & 15) * 8, phase = t >> 4;
    const int rows = q_rows(p, b, i);
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int r0 = phase; r0 < rows; r0 += 32) {
        uint4 gv[4], dv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (r0 + 8 * k < rows) {
                const long long o = tok_off(p, true, b, i * p.tile_q + r0 + 8 * k, h) + e0;
                gv[k] = *reinterpret_cast<const uint4 *>(gate + o);
                dv[k] = *reinterpret_cast<const uint4 *>(dO + o);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (r0 + 8 * k >= rows) break;
            const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w}, dw[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 g2 = unpack2<T>(gw[u]), d2 = unpack2<T>(dw[u]);
                acc[2 * u] = fmaf(g2.x, d2.x, acc[2 * u]);
                acc[2 * u + 1] = fmaf(g2.y, d2.y, acc[2 * u + 1]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) part[phase][e0 + u] = acc[u];
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int ph = 0; ph < 8; ++ph) s += part[ph][t];
    dc[(((long long)b * p.Hq + h) * p.nQ + i) * 128 + t] = s;
}

// Rows: per query tile, A (as in the forward), dA, ds; stores A and ds
// rows [nQ, nKV] per head and dpq = scale ds pk.
__global__ void __launch_bounds__(kCThreads) k_compress_rows(Prob p, const float *__restrict__ pq,
                                                           const float *__restrict__ pk,
                                                           const float *__restrict__ pv,
                                                           const float *__restrict__ dc, float *__restrict__ A,
                                                           float *__restrict__ ds, float *__restrict__ dpq, int qb) {
    extern __shared__ __align__(16) float sm[];
    float *sq = sm;                      // [kCQ][128]
    float *sc = sq + kCQ * 128;          // [kCQ][128] dc rows
    float *sk = sc + kCQ * 128;          // [kCJ][kCPitch] staged pk
    float *sv = sk + kCJ * kCPitch;      // [kCJ][kCPitch] staged pv
    const int pa = nkv_pitch(p);
    float *sA = sv + kCJ * kCPitch;      // [qb][pa] scores, then A
    float *sD = sA + qb * pa;            // [qb][pa] dA, then ds
    const int h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    const int i0 = blockIdx.x * qb, nq = min(qb, p.nQ - i0);
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const long long row0 = ((long long)b * p.Hq + h) * p.nQ + i0;
    const float *pkh = pk + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    const float *pvh = pv + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    float4 fk[4], fv[4];
    chunk_load(fk, pkh, 0, chunk_rows(p.nKV, 0));
    chunk_load(fv, pvh, 0, chunk_rows(p.nKV, 0));
    load_rows(sq, pq + row0 * 128, nq * 128);
    load_rows(sc, dc + row0 * 128, nq * 128);
    for (int j0 = 0; j0 < p.nKV; j0 += kCJ) {
        const int nj = min(kCJ, p.nKV - j0);
        __syncthreads();
        chunk_store(sk, fk, nj);
        chunk_store(sv, fv, nj);
        __syncthreads();
        // the next chunk (after the last one: the dpq pass's first pk chunk)
        const int jn = j0 + kCJ < p.nKV ? j0 + kCJ : 0;
        chunk_load(fk, pkh, jn, chunk_rows(p.nKV, jn));
        if (j0 + kCJ < p.nKV) chunk_load(fv, pvh, jn, chunk_rows(p.nKV, jn));
        if (lane < nj && w < nq) {
            const bool valid = kv_valid(p, b, j0 + lane) > 0;
            const int w2 = min(w + 8, kCQ - 1);
            float s0 = 0.f, s1 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll 2
            for (int d = 0; d < 128; d += 4) {
                const float4 kd = ld4(sk + lane * kCPitch + d), vd = ld4(sv + lane * kCPitch + d);
                s0 = dot4(ld4(sq + w * 128 + d), kd, s0);
                s1 = dot4(ld4(sq + w2 * 128 + d), kd, s1);
                d0 = dot4(ld4(sc + w * 128 + d), vd, d0);
                d1 = dot4(ld4(sc + w2 * 128 + d), vd, d1);
            }
            sA[w * pa + j0 + lane] = valid ? s0 * p.scale : -INFINITY;
            sD[w * pa + j0 + lane] = valid ? d0 : 0.f;
            if (w + 8 < nq) {
                sA[(w + 8) * pa + j0 + lane] = valid ? s1 * p.scale : -INFINITY;
                sD[(w + 8) * pa + j0 + lane] = valid ? d1 : 0.f;
            }
        }
    }
    __syncthreads();
    for (int q = w; q < nq; q += 8) {
        float *ra = sA + q * pa, *rd = sD + q * pa;
        softmax_row(ra, p.nKV, lane);
        float sad = 0.f;
        for (int j = lane; j < p.nKV; j += 32) sad += ra[j] * rd[j];
        sad = warp_sum(sad);
        const long long ro = (row0 + q) * p.nKV;
        for (int j = lane; j < p.nKV; j += 32) {
            const float dsv = ra[j] * (rd[j] - sad);
            rd[j] = dsv;
            A[ro + j] = ra[j];
            ds[ro + j] = dsv;
        }
    }
    // dpq = scale ds pk: thread (dim t % 128, rows 8 (t / 128) .. + 8)
    const int d = t & 127, q0 = (t >> 7) * 8;
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    for (int j0 = 0; j0 < p.nKV; j0 += kCJ) {
        const int nj = min(kCJ, p.nKV - j0);
        __syncthreads();
        chunk_store(sk, fk, nj);
        __syncthreads();
        if (j0 + kCJ < p.nKV) chunk_load(fk, pkh, j0 + kCJ, chunk_rows(p.nKV, j0 + kCJ));
        acc_staged(acc, sD, pa, j0, nj, sk, d, q0, nq);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (q0 + u < nq) dpq[(row0 + q0 + u) * 128 + d] = acc[u] * p.scale;
}

// Columns: CTA (b, key/value head, tiles [j0, j0 + kCJB)): dpv_j = sum A_ij
// dc_i and dpk_j = scale sum ds_ij pq_i over the GQA group's query heads
// (head-major) and query tiles (ascending). Thread: dim t % 128, tiles
// 8 (t / 128) .. + 8.
__global__ void __launch_bounds__(kCThreads) k_compress_cols(Prob p, const float *__restrict__ pq,
                                                           const float *__restrict__ dc,
                                                           const float *__restrict__ A,
                                                           const float *__restrict__ ds, float *__restrict__ dpk,
                                                           float *__restrict__ dpv) {
    __shared__ __align__(16) float spq[kCJ][128];  // filled with 16-byte stores
    __shared__ __align__(16) float sdc[kCJ][128];
    __shared__ float sds[kCJ][kCJB], sa[kCJ][kCJB];
    const int j0 = blockIdx.x * kCJB, hk = blockIdx.y, b = blockIdx.z, g = p.Hq / p.Hkv;
    const int nj = min(kCJB, p.nKV - j0);
    const int t = threadIdx.x, d = t & 127, jg = (t >> 7) * 8;
    float ak[8], av[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) ak[u] = av[u] = 0.f;
    for (int h = hk * g; h < hk * g + g; ++h) {
        const long long base = ((long long)b * p.Hq + h) * p.nQ;
        for (int i0 = 0; i0 < p.nQ; i0 += kCJ) {
            const int ni = min(kCJ, p.nQ - i0);
            __syncthreads();
            load_rows(&spq[0][0], pq + (base + i0) * 128, ni * 128);
            load_rows(&sdc[0][0], dc + (base + i0) * 128, ni * 128);
            for (int x = t; x < ni * kCJB; x += kCThreads) {
                const int ii = x / kCJB, jj = x % kCJB;
                const long long o = (base + i0 + ii) * p.nKV + j0 + jj;
                sds[ii][jj] = jj < nj ? ds[o] : 0.f;
                sa[ii][jj] = jj < nj ? A[o] : 0.f;
            }
            __syncthreads();
            for (int ii = 0; ii < ni; ++ii) {
                const float qv = spq[ii][d], cv = sdc[ii][d];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    ak[u] = fmaf(sds[ii][jg + u], qv, ak[u]);
                    av[u] = fmaf(sa[ii][jg + u], cv, av[u]);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
        if (jg + u < nj) {
            const long long o = (((long long)b * p.Hkv + hk) * p.nKV + j0 + jg + u) * 128 + d;
            dpk[o] = ak[u] * p.scale;
            dpv[o] = av[u];
        }
}

// The row passes' shared memory depends on nKV; their limit is raised to
// what any launch may use, once.
constexpr int kCSmemCap = 200 * 1024;
// Query tiles per CTA of the row passes: the most (up to kCQ) whose score
// rows (rows_per_q floats per tile, per query tile) fit beside the staged
// chunks in 200 KB of shared memory; 0 when not even one fits.
int rows_per_cta(const Prob &p, int fixed_floats, int rows_per_q) {
    for (int qb = kCQ; qb >= 1; qb /= 2)
        if ((size_t)(fixed_floats + (size_t)qb * rows_per_q * nkv_pitch(p)) * 4 <= (size_t)kCSmemCap) return qb;
    return 0;
}

}  // namespace

cudaError_t launch_compress_fwd(const Prob &p, const float *pq, const float *pk, const float *pv, float *c,
                                cudaStream_t s) {
    if (p.nQ == 0 || p.Hq == 0 || p.B == 0) return cudaSuccess;
    const int fixed = kCQ * 128 + kCJ * kCPitch;
    const int qb = rows_per_cta(p, fixed, 1);
    if (qb == 0) return cudaErrorInvalidValue;
    const int smem = (fixed + qb * nkv_pitch(p)) * 4;
    const cudaError_t ae = ensure_smem_limit((const void *)k_compress_fwd, kCSmemCap);
    if (ae != cudaSuccess) return ae;
    dim3 grid((p.nQ + qb - 1) / qb, p.Hq, p.B);
    prof_begin("compress_fwd", s);
    k_compress_fwd<<<grid, kCThreads, smem, s>>>(p, pq, pk, pv, c, qb);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_compress_bwd(const Prob &p, const void *dO, const void *gate, const float *pq, const float *pk,
                                const float *pv, float *dc, float *A, float *ds, float *dpq, float *dpk,
                                float *dpv, cudaStream_t s) {
    if (p.nQ == 0 || p.Hq == 0 || p.B == 0) return cudaSuccess;
    dim3 gq(p.nQ, p.Hq, p.B);
    prof_begin("compress_dc", s);
    if (p.dtype == T_BF16)
        k_compress_dc<__nv_bfloat16><<<gq, 128, 0, s>>>(p, (const __nv_bfloat16 *)dO, (const __nv_bfloat16 *)gate, dc);
    else
        k_compress_dc<__half><<<gq, 128, 0, s>>>(p, (const __half *)dO, (const __half *)gate, dc);
    prof_end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int fixed = 2 * kCQ * 128 + 2 * kCJ * kCPitch;
    const int qb = rows_per_cta(p, fixed, 2);
    if (qb == 0) return cudaErrorInvalidValue;
    const int smem = (fixed + 2 * qb * nkv_pitch(p)) * 4;
    if ((e = ensure_smem_limit((const void *)k_compress_rows, kCSmemCap)) != cudaSuccess) return e;
    dim3 gr((p.nQ + qb - 1) / qb, p.Hq, p.B);
    prof_begin("compress_rows", s);
    k_compress_rows<<<gr, kCThreads, smem, s>>>(p, pq, pk, pv, dc, A, ds, dpq, qb);
    prof_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    dim3 gc((p.nKV + kCJB - 1) / kCJB, p.Hkv, p.B);
    prof_begin("compress_cols", s);
    k_compress_cols<<<gc, kCThreads, 0, s>>>(p, pq, dc, A, ds, dpk, dpv);
    prof_end(s);
    return cudaGetLastError();
}

}  // namespace vsa
