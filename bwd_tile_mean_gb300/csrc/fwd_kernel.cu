// fwd_kernel.cu -- block-sparse attention forward on the 5th-generation
// tensor core (tcgen05, accumulators in TMEM, operands staged by TMA), and
// the forward of the gated compression branch.
//
// Pages: Ascend test_npu_block_sparse_attention_backward.py
// (cpu_block_sparse_attention_tnd_gqa_with_lse: softmax attention over the
// allowed blocks, natural-log LSE, GQA head mapping); FastVideo
// block_sparse_attn_cute_fwd.py (_vbs_mask_mod: key n of tile j is valid iff
// n mod tile < vbs[j]; the forward is Q-owned over the selected KV tiles);
// FastVideo test_vsa256_backward.py (gated compression composes
// out = sparse_out + gate * compress_out without touching sparse_out).
//
// One CTA computes 128 query rows (half of a 256-token video tile, or one
// 128-token block) of one head against its list of selected KV tiles, cut
// into 128-key chunks (chunks without valid keys are skipped). Warp roles:
//   warp 0      builds the chunk list, then one lane issues TMA loads
//               (Q once; K and V per chunk, double-buffered);
//   warp 1      allocates TMEM, then one lane issues the MMAs:
//               S_c = Q K_c^T into one of two TMEM S buffers, and
//               O += P_c V_c into the TMEM O accumulator;
//   warps 4..7  one thread per query row: read S_c from TMEM, mask keys past
//               the chunk's valid count, online softmax in the exp2 domain
//               (rescaling O in TMEM only when the running max grows by more
//               than 2^8), write P_c (16-bit) to shared memory for the PV
//               MMA; finally normalise O, add gate * c when gated, and write
//               O and the LSE.
// TMEM columns: S buffer 0 [0,128), S buffer 1 [128,256), O [256,384).
#include "sm103_ptx.cuh"
#include "vsa_internal.h"

namespace vsa {
using namespace ptx;

namespace {

constexpr int kTile = 32 * 1024;  // one [128 x 128] 16-bit tile = two 64-column TMA boxes
constexpr int kBox = 16 * 1024;
constexpr int kOffQ = 0, kOffK = kTile, kOffV = 3 * kTile, kOffP = 5 * kTile, kOffCtl = 6 * kTile;
constexpr int kCtlBytes = 256 + kMaxChunks * 4 + kMaxChunks * 2;
constexpr size_t kFwdSmem = 1024 + kOffCtl + kCtlBytes;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// Error sites recorded in the device status word.
enum : unsigned { kSiteProd = 0x101, kSiteMma = 0x102, kSiteSoft = 0x103, kSiteEpi = 0x104 };

// S = Q K^T for one 128-key chunk: 8 MMAs of K = 16 along the head dim.
// Q and K tiles are K-major with the 128-byte swizzle; advancing 16
// elements (32 bytes) inside a 64-column box moves the start address.
__device__ __forceinline__ void issue_qk(uint32_t d, uint32_t aQ, uint32_t aK, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
        mma_f16_ss(d, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024), idesc, kk > 0);
    }
}
// O += P V: A = P (K-major over keys), B = V [keys x D] read MN-major
// (D contiguous): 64-wide D halves are LBO = 16 KB apart, 8-key row groups
// SBO = 1 KB apart; each K = 16 step advances 16 keys = 2 KB.
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t aP, uint32_t aV, uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t offp = (kk >> 2) * kBox + (kk & 3) * 32;
        mma_f16_ss(d, sdesc_sw128(aP + offp, 16, 1024), sdesc_sw128(aV + kk * 2048, kBox, 1024), idesc,
                   (acc || kk > 0) ? 1u : 0u);
    }
}

template <typename T>
__global__ void __launch_bounds__(256, 1)
    k_fwd(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
          const __grid_constant__ CUtensorMap tv, const Prob p, const FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sm + kOffQ, *sK = sm + kOffK, *sV = sm + kOffV, *sP = sm + kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffCtl);
    uint64_t *b_q = bars + 0, *b_kf = bars + 1, *b_vf = bars + 3, *b_ke = bars + 5, *b_sf = bars + 7;
    uint64_t *b_pf = bars + 9, *b_od = bars + 10, *b_fin = bars + 11;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 12);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nchunk = reinterpret_cast<int *>(s_tmem + 2);
    int *s_crow = reinterpret_cast<int *>(sm + kOffCtl + 256);
    short *s_cval = reinterpret_cast<short *>(s_crow + kMaxChunks);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int subs = p.tile_q >> 7;
    const int i = blockIdx.x / subs, half = blockIdx.x % subs;
    const int h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    const int row0 = i * p.tile_q + half * 128;
    int nrows = 128;
    if (p.layout == L_TND) {
        nrows = (p.cu_q[b + 1] - p.cu_q[b]) - row0;
        if (nrows <= 0) return;  // whole CTA outside its sequence
        nrows = nrows > 128 ? 128 : nrows;
    }
    const int qrc = (p.layout == L_TND ? p.cu_q[b] : 0) + row0;
    const int kvb = (p.layout == L_TND ? p.cu_kv[b] : 0);
    const int bc = (p.layout == L_TND ? 0 : b);
    const long long qrow = ((long long)b * p.Hq + h) * p.nQ + i;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_kf + s, 1);
            mbar_init(b_vf + s, 1);
            mbar_init(b_ke + s, 1);
            mbar_init(b_sf + s, 1);
        }
        mbar_init(b_pf, 128);
        mbar_init(b_od, 1);
        mbar_init(b_fin, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        // chunk list: (KV row start within the batch entry, valid keys)
        const int cnt = a.q_cnt[qrow];
        const int *idx = a.q_idx + qrow * a.cap;
        const int per = p.tile_kv >> 7;
        int total = 0;
        for (int n0 = 0; n0 < cnt; n0 += 32) {
            const int n = n0 + lane;
            int j = 0, kvv = 0, nc = 0;
            if (n < cnt) {
                j = idx[n];
                kvv = kv_valid(p, b, j);
                nc = min(per, (kvv + 127) >> 7);
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
                if (pos < kMaxChunks) {
                    s_crow[pos] = j * p.tile_kv + c * 128;
                    s_cval[pos] = (short)min(128, kvv - c * 128);
                }
            }
            total += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) *s_nchunk = min(total, kMaxChunks);
    } else if (warp == 1) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *s_tmem;
    const int N = *s_nchunk;
    const bool bf16 = (p.dtype == T_BF16);
    int issued_q = 0, issued[2] = {0, 0}, mma_started = 0;

    if (warp == 0 && lane == 0 && N > 0) {
        // ---------------------------------------------------- TMA producer
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        mbar_expect_tx(b_q, kTile);
        tma_load_4d(sQ, &tq, b_q, 0, qrc, h, bc);
        tma_load_4d(sQ + kBox, &tq, b_q, 64, qrc, h, bc);
        issued_q = 1;
        for (int c = 0; c < N; ++c) {
            const int s = c & 1;
            if (c >= 2 && !mbar_wait(b_ke + s, ((c >> 1) - 1) & 1, s_abort, a.err, kSiteProd)) break;
            const int kr = kvb + s_crow[c];
            mbar_expect_tx(b_kf + s, kTile);
            tma_load_4d(sK + s * kTile, &tk, b_kf + s, 0, kr, hk, bc);
            tma_load_4d(sK + s * kTile + kBox, &tk, b_kf + s, 64, kr, hk, bc);
            mbar_expect_tx(b_vf + s, kTile);
            tma_load_4d(sV + s * kTile, &tv, b_vf + s, 0, kr, hk, bc);
            tma_load_4d(sV + s * kTile + kBox, &tv, b_vf + s, 64, kr, hk, bc);
            issued[s]++;
        }
    } else if (warp == 1 && lane == 0 && N > 0) {
        // ----------------------------------------------------- MMA issuer
        const uint32_t idS = idesc_f16(bf16, 128, 128, false, false);
        const uint32_t idO = idesc_f16(bf16, 128, 128, false, true);
        const uint32_t aQ = smem_addr(sQ), aP = smem_addr(sP), aK = smem_addr(sK), aV = smem_addr(sV);
        bool ok = mbar_wait(b_q, 0, s_abort, a.err, kSiteMma) && mbar_wait(b_kf, 0, s_abort, a.err, kSiteMma);
        if (ok) {
            tc_fence_after();
            issue_qk(tbase, aQ, aK, idS);
            mma_commit(b_sf);
            mma_started = 1;
        }
        for (int c = 0; ok && c < N; ++c) {
            if (c + 1 < N) {
                const int s1 = (c + 1) & 1;
                if (!(ok = mbar_wait(b_kf + s1, ((c + 1) >> 1) & 1, s_abort, a.err, kSiteMma))) break;
                tc_fence_after();
                issue_qk(tbase + s1 * 128, aQ, aK + s1 * kTile, idS);
                mma_commit(b_sf + s1);
            }
            if (!(ok = mbar_wait(b_pf, c & 1, s_abort, a.err, kSiteMma))) break;
            if (!(ok = mbar_wait(b_vf + (c & 1), (c >> 1) & 1, s_abort, a.err, kSiteMma))) break;
            tc_fence_after();
            issue_pv(tbase + 256, aP, aV + (c & 1) * kTile, idO, c > 0);
            mma_commit(b_od);
            mma_commit(b_ke + (c & 1));
        }
    } else if (warp >= 4) {
        // -------------------------------------------- softmax + epilogue
        const int r = (warp - 4) * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)((warp - 4) * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int c = 0; c < N; ++c) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_sf + (c & 1), (c >> 1) & 1, s_abort, a.err, kSiteSoft));
            if (!ok) break;
            tc_fence_after();
            float x[128];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t rr[32];
                tmem_ld32(tl + (c & 1) * 128 + q4 * 32, rr);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) x[q4 * 32 + j] = __uint_as_float(rr[j]);
            }
            const int valid = s_cval[c];
            float mx = -INFINITY;
            if (valid >= 128) {
#pragma unroll
                for (int j = 0; j < 128; ++j) {
                    x[j] *= sl2;
                    mx = fmaxf(mx, x[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 128; ++j) {
                    x[j] = j < valid ? x[j] * sl2 : -INFINITY;
                    mx = fmaxf(mx, x[j]);
                }
            }
            float alpha = 1.f;
            bool resc = false;
            if (c == 0) {
                m_ref = mx;
            } else if (mx > m_ref + 8.f) {
                alpha = ex2(m_ref - mx);
                m_ref = mx;
                resc = true;
            }
            l *= alpha;
            uint32_t pk[64];
            float ls = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float p0 = ex2(x[2 * j] - m_ref), p1 = ex2(x[2 * j + 1] - m_ref);
                ls += p0 + p1;
                pk[j] = pack2<T>(p0, p1);
            }
            l += ls;
            if (c > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(b_od, (c - 1) & 1, s_abort, a.err, kSiteSoft));
                if (!ok) break;
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t o[32];
                    tmem_ld32(tl + 256 + q4 * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(tl + 256 + q4 * 32, o);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    uint4 v;
                    v.x = pk[hf * 32 + u * 4 + 0];
                    v.y = pk[hf * 32 + u * 4 + 1];
                    v.z = pk[hf * 32 + u * 4 + 2];
                    v.w = pk[hf * 32 + u * 4 + 3];
                    *reinterpret_cast<uint4 *>(sP + hf * kBox + sw128_off(r, u)) = v;
                }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(b_pf);
        }
        if (ok && N > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_od, (N - 1) & 1, s_abort, a.err, kSiteEpi));
            if (ok) tc_fence_after();
        }
        const bool have = ok && N > 0;
        const float inv_l = have ? 1.f / l : 0.f;
        const float lse_v = have ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        const bool row_ok = r < nrows;
        const long long ro = tok_off(p, true, b, row0 + r, h);
        T *osp = a.o_sparse ? reinterpret_cast<T *>(a.o_sparse) + ro : nullptr;
        T *out = reinterpret_cast<T *>(a.out) + ro;
        const T *gt = a.gate ? reinterpret_cast<const T *>(a.gate) + ro : nullptr;
        const float *cc = a.gate ? a.c + qrow * 128 : nullptr;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tl + 256 + q4 * 32, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = 0u;
            }
            if (!row_ok) continue;
            float vals[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) vals[j] = __uint_as_float(o[j]) * inv_l;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack2<T>(vals[2 * j], vals[2 * j + 1]);
            if (osp) {
                uint4 *dst = reinterpret_cast<uint4 *>(osp + q4 * 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            }
            if (gt) {
                const uint4 *gsrc = reinterpret_cast<const uint4 *>(gt + q4 * 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 gv = gsrc[u];
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float2 g2 = unpack2<T>(gw[t]);
                        const int e = q4 * 32 + u * 8 + t * 2;
                        w[u * 4 + t] = pack2<T>(vals[u * 8 + t * 2] + g2.x * cc[e],
                                                vals[u * 8 + t * 2 + 1] + g2.y * cc[e + 1]);
                    }
                }
            }
            if (gt || out != osp) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + q4 * 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            }
        }
        if (row_ok && a.lse) a.lse[lse_off(p, b, h, row0 + r)] = lse_v;
    }

    // ------------------------------------------------------------ teardown
    if (*s_abort) {
        // Drain what this CTA started before leaving: outstanding TMA copies
        // (producer) and MMAs (issuer), each with a bounded wait.
        int never = 0;
        if (warp == 0 && lane == 0) {
            if (issued_q) mbar_wait(b_q, 0, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < 2; ++s)
                if (issued[s]) {
                    mbar_wait(b_kf + s, (issued[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
                    mbar_wait(b_vf + s, (issued[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
                }
        }
        if (warp == 1 && lane == 0 && mma_started) {
            mma_commit(b_fin);
            mbar_wait(b_fin, 0, &never, nullptr, 0, 200000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ----------------------------------------------------- compression fwd
// One block per (b, h, query tile): a_j = scale pq . pk_j over non-empty
// KV tiles, A = softmax(a), c[e] = sum_j A_j pv_j[e] (fp32).
__global__ void __launch_bounds__(128) k_compress_fwd(Prob p, const float *__restrict__ pq,
                                                      const float *__restrict__ pk,
                                                      const float *__restrict__ pv, float *__restrict__ c) {
    extern __shared__ float sA[];  // [nKV]
    __shared__ float spq[128];
    __shared__ float red[4];
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const long long row = ((long long)b * p.Hq + h) * p.nQ + i;
    spq[t] = pq[row * 128 + t];
    __syncthreads();
    const float *pkh = pk + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    const float *pvh = pv + ((long long)b * p.Hkv + hk) * p.nKV * 128;
    float mx = -INFINITY;
    for (int j = t; j < p.nKV; j += 128) {
        float x = -INFINITY;
        if (kv_valid(p, b, j) > 0) {
            const float4 *kr = reinterpret_cast<const float4 *>(pkh + (long long)j * 128);
            float acc = 0.f;
#pragma unroll 8
            for (int e = 0; e < 32; ++e) {
                const float4 kv4 = kr[e];
                acc = fmaf(spq[4 * e], kv4.x, acc);
                acc = fmaf(spq[4 * e + 1], kv4.y, acc);
                acc = fmaf(spq[4 * e + 2], kv4.z, acc);
                acc = fmaf(spq[4 * e + 3], kv4.w, acc);
            }
            x = acc * p.scale;
        }
        sA[j] = x;
        mx = fmaxf(mx, x);
    }
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[w] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float sum = 0.f;
    for (int j = t; j < p.nKV; j += 128) {
        const float e = (sA[j] == -INFINITY) ? 0.f : __expf(sA[j] - mx);
        sA[j] = e;
        sum += e;
    }
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) red[w] = sum;
    __syncthreads();
    sum = red[0] + red[1] + red[2] + red[3];
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    float acc = 0.f;
    for (int j = 0; j < p.nKV; ++j) acc = fmaf(sA[j], pvh[(long long)j * 128 + t], acc);
    c[row * 128 + t] = acc * inv;
}

}  // namespace

cudaError_t launch_fwd(const Prob &p, const FwdArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_rows(&tq, p, true, a.q, p.Hq) || !make_tmap_rows(&tk, p, false, a.k, p.Hkv) ||
        !make_tmap_rows(&tv, p, false, a.v, p.Hkv))
        return cudaErrorInvalidValue;
    dim3 grid(p.nQ * (p.tile_q / 128), p.Hq, p.B);
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_fwd<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdSmem);
        cudaFuncSetAttribute(k_fwd<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdSmem);
        attr = true;
    }
    prof_begin("fwd_attn", s);
    if (p.dtype == T_BF16)
        k_fwd<__nv_bfloat16><<<grid, 256, kFwdSmem, s>>>(tq, tk, tv, p, a);
    else
        k_fwd<__half><<<grid, 256, kFwdSmem, s>>>(tq, tk, tv, p, a);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_compress_fwd(const Prob &p, const float *pq, const float *pk, const float *pv, float *c,
                                cudaStream_t s) {
    dim3 grid(p.nQ, p.Hq, p.B);
    if (grid.x == 0) return cudaSuccess;
    prof_begin("compress_fwd", s);
    k_compress_fwd<<<grid, 128, sizeof(float) * p.nKV, s>>>(p, pq, pk, pv, c);
    prof_end(s);
    return cudaGetLastError();
}

}  // namespace vsa
