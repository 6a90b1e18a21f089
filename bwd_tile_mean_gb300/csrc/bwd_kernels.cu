// bwd_kernels.cu -- block-sparse attention backward on tcgen05, plus the
// row-sum preprocess and the gated compression branch's backward.
//
// Pages: Ascend test_npu_block_sparse_attention_backward.py
// (_softmax_backward_np: dS = P (dP - rowsum(P dP)); the TND/GQA backward
// golden: dQ = dS K, dK += dS^T Q, dV += P^T dO, summed over the GQA group);
// FastVideo block_sparse_attn_cute_fwd.py (the backward is KV-owned over
// the transposed index; _CuteAttentionQ128.backward recomputes P from the
// saved LSE with softmax_scale = D^-0.5).
//
// rowsum(P dP) equals Dvec = rowsum(dO * O), computed once per query row
// by k_dvec. The KV-owned pass k_dkdv and the Q-owned pass k_dq each
// recompute S and dP on the tensor core, so neither needs atomics and every
// output element is written by exactly one CTA.
#include "sm103_ptx.cuh"
#include "vsa_internal.h"

namespace vsa {
using namespace ptx;

namespace {

constexpr int kTile = 32 * 1024;
constexpr int kBox = 16 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

enum : unsigned { kSiteDkProd = 0x201, kSiteDkMma = 0x202, kSiteDkSoft = 0x203,
                  kSiteDqProd = 0x301, kSiteDqMma = 0x302, kSiteDqSoft = 0x303 };

// Warp roles of the backward kernels: warps 0-3 and 4-7 are two softmax
// groups (warp w owns TMEM lanes 32*(w%4)..+31); warp 8 issues TMA copies;
// warp 9 owns TMEM and issues the MMAs.
constexpr int kBwdThreads = 320;
constexpr int kProdWarp = 8, kMmaWarp = 9;

// ------------------------------------------------------------------ prep
// Per query slot w of the padded tile layout [B, Hq, nQ * tile_q]:
// lse2[w] = LSE * log2(e) and dvec[w] = sum_d dO_d O_d (rowsum(P dP) of the
// softmax backward). Slots that are not query rows (past a varlen
// sequence's end) get lse2 = +inf and dvec = 0, so P = 0 there. A half-warp
// reads one 256-byte row (16 bytes per lane); each warp keeps four row
// pairs in flight.
template <typename T>
__global__ void __launch_bounds__(256) k_bwd_prep(Prob p, const T *__restrict__ dO, const T *__restrict__ O,
                                                  const float *__restrict__ lse, float *__restrict__ lse2,
                                                  float *__restrict__ dvec) {
    const int per = p.nQ * p.tile_q;
    const long long slots = (long long)p.B * p.Hq * per;
    const int half = (threadIdx.x >> 4) & 1, hl = threadIdx.x & 15;
    const long long wbase = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * 8;
    uint4 av[4], cv[4];
    bool ex[4];
    long long lo[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const long long w = wbase + it * 2 + half;
        ex[it] = false;
        lo[it] = -1;
        av[it] = make_uint4(0, 0, 0, 0);
        cv[it] = make_uint4(0, 0, 0, 0);
        if (w < slots) {
            const int s = (int)(w % per), h = (int)((w / per) % p.Hq), b = (int)(w / ((long long)per * p.Hq));
            ex[it] = p.layout == L_TND ? (s < p.cu_q[b + 1] - p.cu_q[b]) : true;
            if (ex[it]) {
                const long long o = tok_off(p, true, b, s, h) + hl * 8;
                av[it] = __ldg(reinterpret_cast<const uint4 *>(dO + o));
                cv[it] = __ldg(reinterpret_cast<const uint4 *>(O + o));
                lo[it] = lse_off(p, b, h, s);
            }
        }
    }
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const uint32_t aw[4] = {av[it].x, av[it].y, av[it].z, av[it].w};
        const uint32_t cw[4] = {cv[it].x, cv[it].y, cv[it].z, cv[it].w};
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 x = unpack2<T>(aw[u]), y = unpack2<T>(cw[u]);
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const long long w = wbase + it * 2 + half;
        if (hl == 0 && w < slots) {
            dvec[w] = ex[it] ? acc : 0.f;
            lse2[w] = ex[it] ? lse[lo[it]] * kLog2e : INFINITY;
        }
    }
}

// ----------------------------------------------------------- MMA helpers
constexpr int kHalf = 16 * 1024;  // one [64 x 128] 16-bit tile = two 64-column boxes of 8 KB
constexpr int kBox64 = 8 * 1024;

// D = A B^T, A [128 x 128] and B [n x 128] K-major 128-byte-swizzled tiles
// (64-column boxes boxA / boxB bytes apart); 8 MMAs of K = 16.
__device__ __forceinline__ void issue_ss(uint32_t d, uint32_t aA, uint32_t aB, uint32_t idesc, uint32_t boxA,
                                         uint32_t boxB) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t o = (kk & 3) * 32;
        mma_f16_ss(d, sdesc_sw128(aA + (kk >> 2) * boxA + o, 16, 1024), sdesc_sw128(aB + (kk >> 2) * boxB + o, 16, 1024),
                   idesc, kk > 0);
    }
}
// D (+)= A B with A in TMEM (packed 16-bit pairs, 8 columns per K = 16)
// and B [K = 64 rows x N = 128] stored row-major (N contiguous, two 64-
// column boxes of 8 KB), read MN-major; 4 MMAs of K = 16.
__device__ __forceinline__ void issue_ts64(uint32_t d, uint32_t a_tmem, uint32_t aB, uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_f16_ts(d, a_tmem + kk * 8, sdesc_sw128(aB + kk * 2048, kBox64, 1024), idesc, (acc || kk > 0) ? 1u : 0u);
}

// ----------------------------------------------------------------- dK/dV
// One CTA per (b, kv-head hk, 128-key chunk of KV tile j). K and V of the
// chunk stay in shared memory. Work items are 64-row pieces of every query
// tile that selected j, over the query heads of hk's group, in (head,
// ascending tile, piece) order; even items go to softmax group A (warps
// 0-3), odd items to group B (warps 4-7), one thread per key row. Per item:
//   S^T = K Q^T, dP^T = V dO^T           (TMEM, 64 columns each)
//   P^T = exp(scale S^T - LSE_t), dS^T = P^T (dP^T - Dvec_t)
//                                        (packed back into the first 32
//                                         columns of S^T and of dP^T)
//   dV += P^T dO, dK += dS^T Q           (A operands read from TMEM)
// The MMA order S/dP(m), dV/dK(m-1), S/dP(m+1), ... lets one group's
// softmax run while the tensor core works on the other group's item.
// TMEM columns: group A S^T [0,64) dP^T [64,128); group B S^T [128,192)
// dP^T [192,256); dV [256,384); dK [384,512).
constexpr int kDkStages = 4;
constexpr int kDkOffK = 0, kDkOffV = kTile, kDkOffQ = 2 * kTile, kDkOffO = 2 * kTile + kDkStages * kHalf;
constexpr int kDkOffLd = 2 * kTile + 2 * kDkStages * kHalf;  // per stage: lse2[64], dvec[64]
constexpr int kDkOffCtl = kDkOffLd + kDkStages * 512;
constexpr size_t kDkSmem = kDkOffCtl + 256;

struct WorkIter {
    int h, pos, end, sub, i, nsub;
};

__device__ __forceinline__ bool work_next_list(const Prob &p, const BwdArgs &a, int b, int h_end, int j,
                                               WorkIter &w) {
    while (w.pos >= w.end) {
        if (++w.h >= h_end) return false;
        const int *ptr = a.kv_ptr + ((long long)b * p.Hq + w.h) * (p.nKV + 1);
        w.pos = ptr[j];
        w.end = ptr[j + 1];
    }
    w.i = a.kv_qidx[((long long)b * p.Hq + w.h) * p.nQ * a.cap + w.pos];
    w.nsub = (q_rows(p, b, w.i) + 63) >> 6;
    w.sub = 0;
    return true;
}
__device__ __forceinline__ bool work_first(const Prob &p, const BwdArgs &a, int b, int h0, int h_end, int j,
                                           WorkIter &w) {
    w.h = h0;
    const int *ptr = a.kv_ptr + ((long long)b * p.Hq + h0) * (p.nKV + 1);
    w.pos = ptr[j];
    w.end = ptr[j + 1];
    return work_next_list(p, a, b, h_end, j, w);
}
__device__ __forceinline__ bool work_advance(const Prob &p, const BwdArgs &a, int b, int h_end, int j,
                                             WorkIter &w) {
    if (++w.sub < w.nsub) return true;
    ++w.pos;
    return work_next_list(p, a, b, h_end, j, w);
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_dkdv(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
           const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, const Prob p,
           const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    if ((smem_addr(sm) & 1023u) != 0) {  // the swizzled operand tiles need 1024-byte alignment
        if (threadIdx.x == 0) set_error(a.err, 0x2FF);
        return;
    }
    uint8_t *sK = sm + kDkOffK, *sV = sm + kDkOffV, *sQ = sm + kDkOffQ, *sO = sm + kDkOffO, *sLd = sm + kDkOffLd;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kDkOffCtl);
    uint64_t *b_kv = bars + 0, *b_qf = bars + 1, *b_qe = bars + 1 + kDkStages, *b_sf = bars + 1 + 2 * kDkStages;
    uint64_t *b_pd = b_sf + 2, *b_acc = b_sf + 4, *b_fin = b_sf + 5;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(b_sf + 6);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nwork = reinterpret_cast<int *>(s_tmem + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int subs_kv = p.tile_kv >> 7;
    const int j = blockIdx.x / subs_kv, ck = blockIdx.x % subs_kv;
    const int hk = blockIdx.y, b = blockIdx.z, g = p.Hq / p.Hkv;
    const int h0 = hk * g, h_end = h0 + g;
    const int kvalid_tile = kv_valid(p, b, j);
    int kvalid = kvalid_tile - ck * 128;
    kvalid = kvalid < 0 ? 0 : (kvalid > 128 ? 128 : kvalid);
    const int key0 = j * p.tile_kv + ck * 128;  // within the batch entry
    if (p.layout == L_TND && kvalid == 0) return;  // keys outside the sequence do not exist
    const int kvb = (p.layout == L_TND ? p.cu_kv[b] : 0), qb = (p.layout == L_TND ? p.cu_q[b] : 0);
    const int bc = (p.layout == L_TND ? 0 : b);

    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        for (int s = 0; s < kDkStages; ++s) {
            mbar_init(b_qf + s, 1);
            mbar_init(b_qe + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_sf + s, 1);
            mbar_init(b_pd + s, 128);
        }
        mbar_init(b_acc, 1);
        mbar_init(b_fin, 1);
        *s_abort = 0;
        // count the work items (a chunk with no valid key does no work)
        int n = 0;
        if (kvalid > 0)
            for (int h = h0; h < h_end; ++h) {
                const int *ptr = a.kv_ptr + ((long long)b * p.Hq + h) * (p.nKV + 1);
                if (p.layout != L_TND) {  // every query tile has tile_q rows
                    n += (ptr[j + 1] - ptr[j]) * (p.tile_q >> 6);
                    continue;
                }
                const int *lst = a.kv_qidx + ((long long)b * p.Hq + h) * p.nQ * a.cap;
                for (int q = ptr[j]; q < ptr[j + 1]; ++q) n += (q_rows(p, b, lst[q]) + 63) >> 6;
            }
        *s_nwork = n;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *s_tmem;
    const int M = *s_nwork;
    const bool bf16 = (p.dtype == T_BF16);
    int issued_kv = 0, issued[kDkStages] = {0, 0, 0, 0}, mma_started = 0;

    if (warp == kProdWarp && lane == 0 && M > 0) {
        // ------------------------------------------------------ producer
        mbar_expect_tx(b_kv, 2 * kTile);
        tma_load_4d(sK, &tk, b_kv, 0, kvb + key0, hk, bc);
        tma_load_4d(sK + kBox, &tk, b_kv, 64, kvb + key0, hk, bc);
        tma_load_4d(sV, &tv, b_kv, 0, kvb + key0, hk, bc);
        tma_load_4d(sV + kBox, &tv, b_kv, 64, kvb + key0, hk, bc);
        issued_kv = 1;
        WorkIter w;
        bool more = work_first(p, a, b, h0, h_end, j, w);
        for (int m = 0; more && m < M; ++m) {
            const int st = m % kDkStages;
            if (m >= kDkStages && !mbar_wait(b_qe + st, ((m / kDkStages) - 1) & 1, s_abort, a.err, kSiteDkProd))
                break;
            const int row = qb + w.i * p.tile_q + w.sub * 64;
            const long long slot = ((long long)b * p.Hq + w.h) * p.nQ * p.tile_q + w.i * p.tile_q + w.sub * 64;
            mbar_expect_tx(b_qf + st, 2 * kHalf + 512);
            tma_load_4d(sQ + st * kHalf, &tq, b_qf + st, 0, row, w.h, bc);
            tma_load_4d(sQ + st * kHalf + kBox64, &tq, b_qf + st, 64, row, w.h, bc);
            tma_load_4d(sO + st * kHalf, &tdo, b_qf + st, 0, row, w.h, bc);
            tma_load_4d(sO + st * kHalf + kBox64, &tdo, b_qf + st, 64, row, w.h, bc);
            bulk_load(sLd + st * 512, a.lse2 + slot, 256, b_qf + st);
            bulk_load(sLd + st * 512 + 256, a.dvec + slot, 256, b_qf + st);
            issued[st]++;
            more = work_advance(p, a, b, h_end, j, w);
        }
    } else if (warp == kMmaWarp && lane == 0 && M > 0) {
        // ---------------------------------------------------- MMA issuer
        const uint32_t idS = idesc_f16(bf16, 128, 64, false, false);
        const uint32_t idA = idesc_f16(bf16, 128, 128, false, true);
        const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aQ = smem_addr(sQ), aO = smem_addr(sO);
        const uint32_t tS[2] = {tbase, tbase + 128}, tP[2] = {tbase + 64, tbase + 192};
        const uint32_t tdV = tbase + 256, tdK = tbase + 384;
        bool ok = mbar_wait(b_kv, 0, s_abort, a.err, kSiteDkMma);
        for (int m = 0; ok && m < M; ++m) {
            const int st = m % kDkStages, gm = m & 1;
            if (!(ok = mbar_wait(b_qf + st, (m / kDkStages) & 1, s_abort, a.err, kSiteDkMma))) break;
            tc_fence_after();
            issue_ss(tS[gm], aK, aQ + st * kHalf, idS, kBox, kBox64);  // S^T = K Q^T
            issue_ss(tP[gm], aV, aO + st * kHalf, idS, kBox, kBox64);  // dP^T = V dO^T
            mma_commit(b_sf + gm);
            mma_started = 1;
            if (m > 0) {
                const int mp = m - 1, sp = mp % kDkStages, gp = mp & 1;
                if (!(ok = mbar_wait(b_pd + gp, (mp >> 1) & 1, s_abort, a.err, kSiteDkMma))) break;
                tc_fence_after();
                issue_ts64(tdV, tS[gp], aO + sp * kHalf, idA, mp > 0);  // dV += P^T dO
                issue_ts64(tdK, tP[gp], aQ + sp * kHalf, idA, mp > 0);  // dK += dS^T Q
                mma_commit(b_qe + sp);
            }
        }
        if (ok) {
            const int mp = M - 1, sp = mp % kDkStages, gp = mp & 1;
            if (mbar_wait(b_pd + gp, (mp >> 1) & 1, s_abort, a.err, kSiteDkMma)) {
                tc_fence_after();
                issue_ts64(tdV, tS[gp], aO + sp * kHalf, idA, mp > 0);
                issue_ts64(tdK, tP[gp], aQ + sp * kHalf, idA, mp > 0);
                mma_commit(b_qe + sp);
                mma_commit(b_acc);
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------- softmax + epilogue
        const int gw = warp >> 2, lg = warp & 3;  // group, lane quarter
        const int u = lg * 32 + lane;             // key row within the chunk
        const uint32_t tl = tbase + ((uint32_t)(lg * 32) << 16);
        const uint32_t cS = gw * 128, cP = gw * 128 + 64;
        const float sl2 = p.scale * kLog2e;
        const bool key_ok = u < kvalid;
        bool ok = true;
        for (int m = gw; m < M; m += 2) {
            const int st = m % kDkStages;
            ok = __all_sync(0xffffffffu, mbar_wait(b_sf + gw, (m >> 1) & 1, s_abort, a.err, kSiteDkSoft) &&
                                             mbar_wait(b_qf + st, (m / kDkStages) & 1, s_abort, a.err, kSiteDkSoft));
            if (!ok) break;
            tc_fence_after();
            const float4 *sl4 = reinterpret_cast<const float4 *>(sLd + st * 512);
            const float4 *sd4 = reinterpret_cast<const float4 *>(sLd + st * 512 + 256);
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                uint32_t sr[32], dr[32];
                tmem_ld32(tl + cS + q2 * 32, sr);
                tmem_ld32(tl + cP + q2 * 32, dr);
                tmem_wait_ld();
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int t4 = 0; t4 < 8; ++t4) {
                    const float4 l4 = sl4[q2 * 8 + t4], d4 = sd4[q2 * 8 + t4];
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dvv[4] = {d4.x, d4.y, d4.z, d4.w};
                    float pp[4], dd[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float pr = key_ok ? ex2(fmaf(__uint_as_float(sr[t4 * 4 + e]), sl2, -lv[e])) : 0.f;
                        pp[e] = pr;
                        dd[e] = pr * (__uint_as_float(dr[t4 * 4 + e]) - dvv[e]);
                    }
                    pw[t4 * 2] = pack2<T>(pp[0], pp[1]);
                    pw[t4 * 2 + 1] = pack2<T>(pp[2], pp[3]);
                    dw[t4 * 2] = pack2<T>(dd[0], dd[1]);
                    dw[t4 * 2 + 1] = pack2<T>(dd[2], dd[3]);
                }
                tmem_st16(tl + cS + q2 * 16, pw);  // P^T over S^T's consumed columns
                tmem_st16(tl + cP + q2 * 16, dw);  // dS^T over dP^T's consumed columns
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_pd + gw);
        }
        if (ok && M > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_acc, 0, s_abort, a.err, kSiteDkSoft));
            if (ok) tc_fence_after();
        }
        const bool have = ok && M > 0;
        const bool row_ok = (p.layout == L_TND) ? key_ok : true;
        const long long ro = tok_off(p, false, b, key0 + u, hk);
        T *dst = reinterpret_cast<T *>(gw ? a.dk : a.dv) + ro;   // group A writes dV, group B dK
        const float inv = kvalid_tile > 0 ? 1.f / (float)kvalid_tile : 0.f;
        const float *cbase = gw ? a.dpk : a.dpv;
        const float *cadd = cbase ? cbase + (((long long)b * p.Hkv + hk) * p.nKV + j) * 128 : nullptr;
        const float mul = gw ? p.scale : 1.f;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tl + 256 + gw * 128 + q4 * 32, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (!row_ok) continue;
            uint32_t wv[16];
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
                float v0 = key_ok ? __uint_as_float(o[2 * e2]) * mul : 0.f;
                float v1 = key_ok ? __uint_as_float(o[2 * e2 + 1]) * mul : 0.f;
                if (cadd && key_ok) {
                    v0 += cadd[q4 * 32 + 2 * e2] * inv;
                    v1 += cadd[q4 * 32 + 2 * e2 + 1] * inv;
                }
                wv[e2] = pack2<T>(v0, v1);
            }
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + q4 * 32);
#pragma unroll
            for (int t = 0; t < 4; ++t) d4[t] = make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
        }
    }

    if (*s_abort) {
        int never = 0;
        if (warp == kProdWarp && lane == 0) {
            if (issued_kv) mbar_wait(b_kv, 0, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < kDkStages; ++s)
                if (issued[s]) mbar_wait(b_qf + s, (issued[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
        }
        if (warp == kMmaWarp && lane == 0 && mma_started) {
            mma_commit(b_fin);
            mbar_wait(b_fin, 0, &never, nullptr, 0, 200000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// -------------------------------------------------------------------- dQ
// One CTA per (b, h, query tile i): two groups of 128 rows (A: warps 0-3,
// B: warps 4-7; one group for 128-token tiles) share 64-key chunks of the
// selected KV tiles. Per chunk and group:
//   S = Q K^T, dP = dO V^T                 (TMEM, 64 columns each)
//   dS = P (dP - Dvec), P = exp(scale S - LSE)
//                                          (packed into S's first 32 columns)
//   dQ += dS K                             (A operand read from TMEM)
// MMA order per chunk c: S/dP_A(c), dQ_B(c-1), S/dP_B(c), dQ_A(c).
// TMEM columns: group A S [0,64) dP [64,128); group B S [128,192)
// dP [192,256); dQ_A [256,384); dQ_B [384,512).
constexpr int kDqOffQ = 0, kDqOffO = 2 * kTile, kDqOffK = 4 * kTile, kDqOffV = 4 * kTile + 2 * kHalf;
constexpr int kDqOffCtl = 6 * kTile;
constexpr size_t kDqSmem = kDqOffCtl + 256 + kMaxChunks64 * 6;

template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_dq(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
         const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, const Prob p,
         const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    if ((smem_addr(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) set_error(a.err, 0x3FF);
        return;
    }
    uint8_t *sQ = sm + kDqOffQ, *sO = sm + kDqOffO, *sK = sm + kDqOffK, *sV = sm + kDqOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kDqOffCtl);
    uint64_t *b_q = bars + 0, *b_kf = bars + 1, *b_ke = bars + 3, *b_vf = bars + 5, *b_ve = bars + 7;
    uint64_t *b_sf = bars + 9, *b_dsf = bars + 11, *b_dq = bars + 13, *b_fin = bars + 15;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nchunk = reinterpret_cast<int *>(s_tmem + 2);
    int *s_crow = reinterpret_cast<int *>(sm + kDqOffCtl + 256);
    short *s_cval = reinterpret_cast<short *>(s_crow + kMaxChunks64);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    int nrows[2];
    for (int gg = 0; gg < 2; ++gg) {
        const int r0 = i * p.tile_q + gg * 128;
        int n = (gg * 128 < p.tile_q) ? 128 : 0;
        if (p.layout == L_TND && n > 0) {
            n = (p.cu_q[b + 1] - p.cu_q[b]) - r0;
            n = n < 0 ? 0 : (n > 128 ? 128 : n);
        }
        nrows[gg] = n;
    }
    if (nrows[0] == 0) return;
    const bool has_b = nrows[1] > 0;
    const int qbase = (p.layout == L_TND ? p.cu_q[b] : 0) + i * p.tile_q;
    const int kvb = (p.layout == L_TND ? p.cu_kv[b] : 0);
    const int bc = (p.layout == L_TND ? 0 : b);
    const long long qrow = ((long long)b * p.Hq + h) * p.nQ + i;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_kf + s, 1);
            mbar_init(b_ke + s, 1);
            mbar_init(b_vf + s, 1);
            mbar_init(b_ve + s, 1);
            mbar_init(b_sf + s, 1);
            mbar_init(b_dsf + s, 128);
            mbar_init(b_dq + s, 1);
        }
        mbar_init(b_fin, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == kProdWarp) {
        // chunk list of 64-key chunks: (KV row start within the batch entry, valid keys)
        const int cnt = a.q_cnt[qrow];
        const int *idx = a.q_idx + qrow * a.cap;
        const int per = p.tile_kv >> 6;
        int total = 0;
        for (int n0 = 0; n0 < cnt; n0 += 32) {
            const int n = n0 + lane;
            int jj = 0, kvv = 0, nc = 0;
            if (n < cnt) {
                jj = idx[n];
                kvv = kv_valid(p, b, jj);
                nc = min(per, (kvv + 63) >> 6);
            }
            int inc = nc;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += y;
            }
            const int base = total + inc - nc;
            for (int c = 0; c < nc; ++c) {
                const int pos = base + c;
                if (pos < kMaxChunks64) {
                    s_crow[pos] = jj * p.tile_kv + c * 64;
                    s_cval[pos] = (short)min(64, kvv - c * 64);
                }
            }
            total += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) *s_nchunk = min(total, kMaxChunks64);
    } else if (warp == kMmaWarp) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *s_tmem;
    const int N = *s_nchunk;
    const bool bf16 = (p.dtype == T_BF16);
    int issued_q = 0, issued_k[2] = {0, 0}, issued_v[2] = {0, 0}, mma_started = 0;

    if (warp == kProdWarp && lane == 0 && N > 0) {
        const int ng = has_b ? 2 : 1;
        mbar_expect_tx(b_q, ng * 2 * kTile);
        for (int gg = 0; gg < ng; ++gg) {
            tma_load_4d(sQ + gg * kTile, &tq, b_q, 0, qbase + gg * 128, h, bc);
            tma_load_4d(sQ + gg * kTile + kBox, &tq, b_q, 64, qbase + gg * 128, h, bc);
            tma_load_4d(sO + gg * kTile, &tdo, b_q, 0, qbase + gg * 128, h, bc);
            tma_load_4d(sO + gg * kTile + kBox, &tdo, b_q, 64, qbase + gg * 128, h, bc);
        }
        issued_q = 1;
        for (int c = 0; c < N; ++c) {
            const int s = c & 1;
            const int kr = kvb + s_crow[c];
            if (c >= 2 && !mbar_wait(b_ke + s, ((c >> 1) - 1) & 1, s_abort, a.err, kSiteDqProd)) break;
            mbar_expect_tx(b_kf + s, kHalf);
            tma_load_4d(sK + s * kHalf, &tk, b_kf + s, 0, kr, hk, bc);
            tma_load_4d(sK + s * kHalf + kBox64, &tk, b_kf + s, 64, kr, hk, bc);
            issued_k[s]++;
            if (c >= 2 && !mbar_wait(b_ve + s, ((c >> 1) - 1) & 1, s_abort, a.err, kSiteDqProd)) break;
            mbar_expect_tx(b_vf + s, kHalf);
            tma_load_4d(sV + s * kHalf, &tv, b_vf + s, 0, kr, hk, bc);
            tma_load_4d(sV + s * kHalf + kBox64, &tv, b_vf + s, 64, kr, hk, bc);
            issued_v[s]++;
        }
    } else if (warp == kMmaWarp && lane == 0 && N > 0) {
        const uint32_t idS = idesc_f16(bf16, 128, 64, false, false);
        const uint32_t idQ = idesc_f16(bf16, 128, 128, false, true);
        const uint32_t aQ = smem_addr(sQ), aO = smem_addr(sO), aK = smem_addr(sK), aV = smem_addr(sV);
        const uint32_t tS[2] = {tbase, tbase + 128}, tP[2] = {tbase + 64, tbase + 192};
        const uint32_t tQ[2] = {tbase + 256, tbase + 384};
        bool ok = mbar_wait(b_q, 0, s_abort, a.err, kSiteDqMma);
        for (int c = 0; ok && c < N; ++c) {
            const int s = c & 1, sp = (c - 1) & 1;
            if (!(ok = mbar_wait(b_kf + s, (c >> 1) & 1, s_abort, a.err, kSiteDqMma))) break;
            if (!(ok = mbar_wait(b_vf + s, (c >> 1) & 1, s_abort, a.err, kSiteDqMma))) break;
            tc_fence_after();
            issue_ss(tS[0], aQ, aK + s * kHalf, idS, kBox, kBox64);  // S_A = Q_A K^T
            issue_ss(tP[0], aO, aV + s * kHalf, idS, kBox, kBox64);  // dP_A = dO_A V^T
            mma_commit(b_sf + 0);
            mma_started = 1;
            if (has_b) {
                if (c > 0) {
                    if (!(ok = mbar_wait(b_dsf + 1, (c - 1) & 1, s_abort, a.err, kSiteDqMma))) break;
                    tc_fence_after();
                    issue_ts64(tQ[1], tS[1], aK + sp * kHalf, idQ, c - 1 > 0);  // dQ_B += dS_B K
                    mma_commit(b_dq + 1);
                    mma_commit(b_ke + sp);
                }
                issue_ss(tS[1], aQ + kTile, aK + s * kHalf, idS, kBox, kBox64);
                issue_ss(tP[1], aO + kTile, aV + s * kHalf, idS, kBox, kBox64);
                mma_commit(b_sf + 1);
            }
            mma_commit(b_ve + s);
            if (!(ok = mbar_wait(b_dsf + 0, c & 1, s_abort, a.err, kSiteDqMma))) break;
            tc_fence_after();
            issue_ts64(tQ[0], tS[0], aK + s * kHalf, idQ, c > 0);  // dQ_A += dS_A K
            mma_commit(b_dq + 0);
            if (!has_b) mma_commit(b_ke + s);
        }
        if (ok && has_b) {
            const int sp = (N - 1) & 1;
            if (mbar_wait(b_dsf + 1, (N - 1) & 1, s_abort, a.err, kSiteDqMma)) {
                tc_fence_after();
                issue_ts64(tQ[1], tS[1], aK + sp * kHalf, idQ, N - 1 > 0);
                mma_commit(b_dq + 1);
                mma_commit(b_ke + sp);
            }
        }
    } else if (warp < 8 && (warp < 4 || has_b)) {
        const int gw = warp >> 2, lg = warp & 3;
        const int r = lg * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(lg * 32) << 16);
        const uint32_t cS = gw * 128, cP = gw * 128 + 64, cQ = 256 + gw * 128;
        const float sl2 = p.scale * kLog2e;
        const bool row_ok = r < nrows[gw];
        const int row = i * p.tile_q + gw * 128 + r;  // within the batch entry
        const long long slot = ((long long)b * p.Hq + h) * p.nQ * p.tile_q + row;
        const float l2 = N > 0 ? a.lse2[slot] : INFINITY;
        const float dvv = N > 0 ? a.dvec[slot] : 0.f;
        bool ok = true;
        for (int c = 0; c < N; ++c) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_sf + gw, c & 1, s_abort, a.err, kSiteDqSoft));
            if (!ok) break;
            tc_fence_after();
            const int valid = s_cval[c];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                uint32_t sr[32], dr[32];
                tmem_ld32(tl + cS + q2 * 32, sr);
                tmem_ld32(tl + cP + q2 * 32, dr);
                tmem_wait_ld();
                uint32_t dw[16];
#pragma unroll
                for (int t2 = 0; t2 < 16; ++t2) {
                    float dd[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kk = q2 * 32 + t2 * 2 + e;
                        const float pr = kk < valid ? ex2(fmaf(__uint_as_float(sr[t2 * 2 + e]), sl2, -l2)) : 0.f;
                        dd[e] = pr * (__uint_as_float(dr[t2 * 2 + e]) - dvv);
                    }
                    dw[t2] = pack2<T>(dd[0], dd[1]);
                }
                tmem_st16(tl + cS + q2 * 16, dw);  // dS over S's consumed columns
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_dsf + gw);
        }
        if (ok && N > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_dq + gw, (N - 1) & 1, s_abort, a.err, kSiteDqSoft));
            if (ok) tc_fence_after();
        }
        const bool have = ok && N > 0;
        const long long ro = tok_off(p, true, b, row, h);
        T *dq = reinterpret_cast<T *>(a.dq) + ro;
        const int qv = a.dpq ? q_valid(p, b, i) : 0;
        const bool add_c = a.dpq && (gw * 128 + r) < qv;
        const float *cq = a.dpq ? a.dpq + qrow * 128 : nullptr;
        const float inv = qv > 0 ? 1.f / (float)qv : 0.f;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tl + cQ + q4 * 32, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (!row_ok) continue;
            uint32_t wv[16];
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
                float v0 = __uint_as_float(o[2 * e2]) * p.scale, v1 = __uint_as_float(o[2 * e2 + 1]) * p.scale;
                if (add_c) {
                    v0 += cq[q4 * 32 + 2 * e2] * inv;
                    v1 += cq[q4 * 32 + 2 * e2 + 1] * inv;
                }
                wv[e2] = pack2<T>(v0, v1);
            }
            uint4 *d4 = reinterpret_cast<uint4 *>(dq + q4 * 32);
#pragma unroll
            for (int t = 0; t < 4; ++t) d4[t] = make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
        }
    }

    if (*s_abort) {
        int never = 0;
        if (warp == kProdWarp && lane == 0) {
            if (issued_q) mbar_wait(b_q, 0, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < 2; ++s) {
                if (issued_k[s]) mbar_wait(b_kf + s, (issued_k[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
                if (issued_v[s]) mbar_wait(b_vf + s, (issued_v[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
            }
        }
        if (warp == kMmaWarp && lane == 0 && mma_started) {
            mma_commit(b_fin);
            mbar_wait(b_fin, 0, &never, nullptr, 0, 200000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// --------------------------------------------------- compression backward
// dc_i = sum over the query rows of tile i of gate (*) dO (fp32, per dim).
template <typename T>
__global__ void __launch_bounds__(128) k_compress_dc(Prob p, const T *__restrict__ dO, const T *__restrict__ gate,
                                                     float *__restrict__ dc) {
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, e = threadIdx.x;
    const int rows = q_rows(p, b, i);
    float acc = 0.f;
    for (int t = 0; t < rows; ++t) {
        const long long o = tok_off(p, true, b, i * p.tile_q + t, h) + e;
        acc = fmaf(to_f<T>(gate[o]), to_f<T>(dO[o]), acc);
    }
    dc[(((long long)b * p.Hq + h) * p.nQ + i) * 128 + e] = acc;
}

// Per query tile: A_j (softmax over non-empty KV tiles of scale pq.pk_j),
// dA_j = dc . pv_j, ds_j = A_j (dA_j - sum A dA); stores A and ds, and
// dpq = scale sum_j ds_j pk_j.
__global__ void __launch_bounds__(128) k_compress_rows(Prob p, const float *__restrict__ pq,
                                                       const float *__restrict__ pk, const float *__restrict__ pv,
                                                       const float *__restrict__ dc, float *__restrict__ A,
                                                       float *__restrict__ ds, float *__restrict__ dpq) {
    extern __shared__ float sh[];  // sA[nKV], sD[nKV]
    float *sA = sh, *sD = sh + p.nKV;
    __shared__ float spq[128], sdc[128], red[4];
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const long long row = ((long long)b * p.Hq + h) * p.nQ + i;
    spq[t] = pq[row * 128 + t];
    sdc[t] = dc[row * 128 + t];
    __syncthreads();
    const float *pkh = pk + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    const float *pvh = pv + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    float mx = -INFINITY;
    for (int j = t; j < p.nKV; j += 128) {
        float x = -INFINITY, da = 0.f;
        if (kv_valid(p, b, j) > 0) {
            float acc = 0.f, acc2 = 0.f;
            for (int e = 0; e < 128; ++e) {
                acc = fmaf(spq[e], pkh[(long long)j * 128 + e], acc);
                acc2 = fmaf(sdc[e], pvh[(long long)j * 128 + e], acc2);
            }
            x = acc * p.scale;
            da = acc2;
        }
        sA[j] = x;
        sD[j] = da;
        mx = fmaxf(mx, x);
    }
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[w] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float sum = 0.f;
    for (int j = t; j < p.nKV; j += 128) {
        const float ev = sA[j] == -INFINITY ? 0.f : __expf(sA[j] - mx);
        sA[j] = ev;
        sum += ev;
    }
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) red[w] = sum;
    __syncthreads();
    sum = red[0] + red[1] + red[2] + red[3];
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    __syncthreads();
    float sad = 0.f;
    for (int j = t; j < p.nKV; j += 128) {
        sA[j] *= inv;
        sad += sA[j] * sD[j];
    }
    for (int off = 16; off > 0; off >>= 1) sad += __shfl_xor_sync(0xffffffffu, sad, off);
    if (lane == 0) red[w] = sad;
    __syncthreads();
    sad = red[0] + red[1] + red[2] + red[3];
    for (int j = t; j < p.nKV; j += 128) {
        const float d = sA[j] * (sD[j] - sad);
        sD[j] = d;
        A[row * p.nKV + j] = sA[j];
        ds[row * p.nKV + j] = d;
    }
    __syncthreads();
    float acc = 0.f;
    for (int j = 0; j < p.nKV; ++j) acc = fmaf(sD[j], pkh[(long long)j * 128 + t], acc);
    dpq[row * 128 + t] = acc * p.scale;
}

// Per KV tile: dpv_j = sum_{h in group, i} A_ij dc_i and
// dpk_j = scale sum_{h, i} ds_ij pq_i.
__global__ void __launch_bounds__(128) k_compress_cols(Prob p, const float *__restrict__ pq,
                                                       const float *__restrict__ dc, const float *__restrict__ A,
                                                       const float *__restrict__ ds, float *__restrict__ dpk,
                                                       float *__restrict__ dpv) {
    const int j = blockIdx.x, hk = blockIdx.y, b = blockIdx.z, e = threadIdx.x, g = p.Hq / p.Hkv;
    float ak = 0.f, av = 0.f;
    for (int h = hk * g; h < hk * g + g; ++h) {
        const long long base = ((long long)b * p.Hq + h) * p.nQ;
        for (int i = 0; i < p.nQ; ++i) {
            const long long row = base + i;
            ak = fmaf(ds[row * p.nKV + j], pq[row * 128 + e], ak);
            av = fmaf(A[row * p.nKV + j], dc[row * 128 + e], av);
        }
    }
    const long long o = (((long long)b * p.Hkv + hk) * p.nKV + j) * 128 + e;
    dpk[o] = ak * p.scale;
    dpv[o] = av;
}

}  // namespace

cudaError_t launch_bwd_prep(const Prob &p, const void *dO, const void *o, const float *lse, float *lse2,
                            float *dvec, cudaStream_t s) {
    const long long slots = (long long)p.B * p.Hq * p.nQ * p.tile_q;
    if (slots == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((slots + 63) / 64);
    prof_begin("bwd_prep", s);
    if (p.dtype == T_BF16)
        k_bwd_prep<__nv_bfloat16><<<blocks, 256, 0, s>>>(p, (const __nv_bfloat16 *)dO, (const __nv_bfloat16 *)o,
                                                        lse, lse2, dvec);
    else
        k_bwd_prep<__half><<<blocks, 256, 0, s>>>(p, (const __half *)dO, (const __half *)o, lse, lse2, dvec);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const Prob &p, const BwdArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv, tdo;  // q / dO in 64-row boxes, k / v in 128-row boxes
    if (!make_tmap_rows(&tq, p, true, a.q, p.Hq, 64) || !make_tmap_rows(&tk, p, false, a.k, p.Hkv, 128) ||
        !make_tmap_rows(&tv, p, false, a.v, p.Hkv, 128) || !make_tmap_rows(&tdo, p, true, a.dO, p.Hq, 64))
        return cudaErrorInvalidValue;
    dim3 grid(p.nKV * (p.tile_kv / 128), p.Hkv, p.B);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_dkdv<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDkSmem);
        cudaFuncSetAttribute(k_dkdv<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDkSmem);
        attr = true;
    }
    prof_begin("bwd_dkdv", s);
    if (p.dtype == T_BF16)
        k_dkdv<__nv_bfloat16><<<grid, kBwdThreads, kDkSmem, s>>>(tq, tk, tv, tdo, p, a);
    else
        k_dkdv<__half><<<grid, kBwdThreads, kDkSmem, s>>>(tq, tk, tv, tdo, p, a);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const Prob &p, const BwdArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv, tdo;  // q / dO in 128-row boxes, k / v in 64-row boxes
    if (!make_tmap_rows(&tq, p, true, a.q, p.Hq, 128) || !make_tmap_rows(&tk, p, false, a.k, p.Hkv, 64) ||
        !make_tmap_rows(&tv, p, false, a.v, p.Hkv, 64) || !make_tmap_rows(&tdo, p, true, a.dO, p.Hq, 128))
        return cudaErrorInvalidValue;
    dim3 grid(p.nQ, p.Hq, p.B);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_dq<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDqSmem);
        cudaFuncSetAttribute(k_dq<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDqSmem);
        attr = true;
    }
    prof_begin("bwd_dq", s);
    if (p.dtype == T_BF16)
        k_dq<__nv_bfloat16><<<grid, kBwdThreads, kDqSmem, s>>>(tq, tk, tv, tdo, p, a);
    else
        k_dq<__half><<<grid, kBwdThreads, kDqSmem, s>>>(tq, tk, tv, tdo, p, a);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_compress_bwd(const Prob &p, const void *dO, const void *gate, const float *pq, const float *pk,
                                const float *pv, float *dc, float *A, float *ds, float *dpq, float *dpk,
                                float *dpv, cudaStream_t s) {
    dim3 gq(p.nQ, p.Hq, p.B), gk(p.nKV, p.Hkv, p.B);
    prof_begin("compress_dc", s);
    if (p.dtype == T_BF16)
        k_compress_dc<__nv_bfloat16><<<gq, 128, 0, s>>>(p, (const __nv_bfloat16 *)dO, (const __nv_bfloat16 *)gate, dc);
    else
        k_compress_dc<__half><<<gq, 128, 0, s>>>(p, (const __half *)dO, (const __half *)gate, dc);
    prof_end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prof_begin("compress_rows", s);
    k_compress_rows<<<gq, 128, sizeof(float) * 2 * p.nKV, s>>>(p, pq, pk, pv, dc, A, ds, dpq);
    prof_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prof_begin("compress_cols", s);
    k_compress_cols<<<gk, 128, 0, s>>>(p, pq, dc, A, ds, dpk, dpv);
    prof_end(s);
    return cudaGetLastError();
}

}  // namespace vsa
