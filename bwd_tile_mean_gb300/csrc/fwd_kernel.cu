// fwd_kernel.cu -- block-sparse attention forward on the 5th-generation
// tensor core (tcgen05, accumulators in TMEM, operands staged by TMA); the
// gated compression branch's c comes from compress_kernels.cu and is added
// in the epilogue.
//
// Pages: Ascend test_npu_block_sparse_attention_backward.py
// (cpu_block_sparse_attention_tnd_gqa_with_lse: softmax attention over the
// allowed blocks, natural-log LSE, GQA head mapping); FastVideo
// block_sparse_attn_cute_fwd.py (_vbs_mask_mod: key n of tile j is valid iff
// n mod tile < vbs[j]; the forward is Q-owned over the selected KV tiles);
// FastVideo test_vsa256_backward.py (gated compression composes
// out = sparse_out + gate * compress_out without touching sparse_out).
//
// 256-token query tiles without query-block masks run on CTA pairs
// (k_fwd2, further down); the single-CTA kernel k_fwd described here takes
// 128-token tiles, tiles with query-block masks, and the tiles k_fwd2 hands
// back for a recompute.
//
// One CTA computes one query tile: two groups of 128 rows (A and B; the
// two halves of a 256-token video tile, or a single group for 128-token
// tiles) of one head against the tile's selected KV tiles, cut into
// 128-key chunks (chunks without valid keys are skipped). Both groups share
// every K/V chunk. Warp roles:
//   warps 0-3   softmax of group A, one thread per query row;
//   warps 4-7   softmax of group B;
//   warp 8      builds the chunk list, then one lane issues TMA loads
//               (Q of both groups once; K and V per chunk, two stages);
//   warp 9      allocates TMEM, then one lane issues the MMAs.
// Per chunk c the MMAs go S_A(c) = Q_A K_c^T, O_B += P_B(c-1) V_(c-1),
// S_B(c) = Q_B K_c^T, O_A += P_A(c) V_c, so each group's softmax runs while
// the tensor core works for the other group. The softmax loads a whole row
// of S (128 scores) from TMEM with one wait and computes probabilities in
// the exp2 domain against the row's running reference (keys past the
// chunk's valid count masked; scale-and-subtract and the row sum on paired
// f32 instructions). The row max is taken only on the first chunk and when
// a chunk's row sum shows that an element grew past the 16-bit operand's
// safe range; only then does the reference move (when the max is more than
// 2^8 above it) and l and O get rescaled in TMEM. P goes back into the first
// 64 columns of the S buffer as packed 16-bit pairs; the PV MMA reads it as
// its A operand. The epilogue normalises O, adds gate * c
// when gated, and writes O and the LSE.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
#include "sm103_ptx.cuh"
#include "vsa_internal.h"

namespace vsa {
using namespace ptx;

namespace {

constexpr int kTile = 32 * 1024;  // one [128 x 128] 16-bit tile = two 64-column TMA boxes
constexpr int kBox = 16 * 1024;
constexpr int kOffQ = 0, kOffK = 2 * kTile, kOffV = 4 * kTile, kOffCtl = 6 * kTile;
constexpr int kCtlBytes = 256 + kMaxChunks * 4 + kMaxChunks * 2 + kMaxChunks * 4;
constexpr size_t kFwdSmem = kOffCtl + kCtlBytes;
constexpr int kFwdThreads = 320;
constexpr int kFwdProdWarp = 8, kFwdMmaWarp = 9;
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
        mma_f16_ss_w(d, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024), idesc, kk > 0);
    }
}
// O += P V: A = P in TMEM (128 keys = 64 packed columns, 8 per K = 16
// step), B = V [keys x D] read MN-major (D contiguous): 64-wide D halves
// are LBO = 16 KB apart, 8-key row groups SBO = 1 KB apart; each K = 16
// step advances 16 keys = 2 KB.
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t p_tmem, uint32_t aV, uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_f16_ts_w(d, p_tmem + kk * 8, sdesc_sw128(aV + kk * 2048, kBox, 1024), idesc, (acc || kk > 0) ? 1u : 0u);
}

// Bound on a row's chunk sum of probabilities that keeps every element a
// finite 16-bit operand of the PV MMA: bf16 shares fp32's exponent range,
// fp16 ends at 65504.
template <typename T> struct SumLimit;
template <> struct SumLimit<__nv_bfloat16> { static constexpr float value = 0x1p64f; };
template <> struct SumLimit<__half> { static constexpr float value = 0x1p15f; };

// P = exp2(scale log2e s - m) for the 128 scores of one row (or the 32-key
// quarters [Q0, Q1) of them), packed to 16-bit pairs into the 64 TMEM
// columns at taddr; returns the fp32 row sum of those keys
// (scale-and-subtract and the sum on paired f32 instructions).
template <typename T, int Q0 = 0, int Q1 = 4>
__device__ __forceinline__ float exp_row(const uint32_t (&sr)[128], float m, float sl2, uint32_t taddr) {
    const uint64_t sc2 = f32x2(sl2, sl2), nm2 = f32x2(-m, -m);
    uint64_t acc0 = f32x2(0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int q4 = Q0; q4 < Q1; ++q4) {
        uint32_t w16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int e = q4 * 32 + 2 * j;
            const float2 x =
                f32x2_split(ffma_x2(f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2, nm2));
            const float p0 = ex2(x.x), p1 = ex2(x.y);
            if (j & 1)
                acc1 = fadd_x2(acc1, f32x2(p0, p1));
            else
                acc0 = fadd_x2(acc0, f32x2(p0, p1));
            w16[j] = pack2<T>(p0, p1);
        }
        tmem_st16(taddr + q4 * 16, w16);
    }
    const float2 s0 = f32x2_split(acc0), s1 = f32x2_split(acc1);
    return (s0.x + s0.y) + (s1.x + s1.y);
}

constexpr int kRedoGroup = 16;  // query tiles of one head per CTA of the redo launch
constexpr int kFwdBars = 16;

// One query tile (i, h, b) with the CTA's TMEM columns at *s_tmem (512 of
// them, allocated by the kernel); its barriers are initialised here and
// invalidated on the way out, so the next tile of the same CTA starts from
// fresh ones.
template <typename T>
__device__ __forceinline__ void fwd_tile(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                         const Prob &p, const FwdArgs &a, uint8_t *sm, int i, int h, int b) {
    uint8_t *sQ = sm + kOffQ, *sK = sm + kOffK, *sV = sm + kOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffCtl);
    uint64_t *b_q = bars + 0, *b_kf = bars + 1, *b_vf = bars + 3, *b_ke = bars + 5, *b_sf = bars + 7;
    uint64_t *b_pf = bars + 9, *b_od = bars + 11, *b_fin = bars + 13, *b_ve = bars + 14;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nchunk = reinterpret_cast<int *>(s_tmem + 2);
    int *s_crow = reinterpret_cast<int *>(sm + kOffCtl + 256);
    short *s_cval = reinterpret_cast<short *>(s_crow + kMaxChunks);
    int *s_csub = reinterpret_cast<int *>(s_cval + kMaxChunks);  // query-block bits of each chunk's tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hk = h / (p.Hq / p.Hkv);
    // rows of each 128-row group (0 if the group does not exist)
    int nrows[2];
    for (int g = 0; g < 2; ++g) {
        const int r0 = i * p.tile_q + g * 128;
        int n = (g * 128 < p.tile_q) ? 128 : 0;
        if (p.layout == L_TND && n > 0) {
            n = seq_len(p, true, b) - r0;
            n = n < 0 ? 0 : (n > 128 ? 128 : n);
        }
        nrows[g] = n;
    }
    if (nrows[0] == 0) return;  // the whole tile lies outside its sequence
    const bool has_b = nrows[1] > 0;
    const int qbase = (p.layout == L_TND ? seq_start(p, true, b) : 0) + i * p.tile_q;
    const int kvb = (p.layout == L_TND ? seq_start(p, false, b) : 0);
    const int bc = (p.layout == L_TND ? 0 : b);
    const long long qrow = ((long long)b * p.Hq + h) * p.nQ + i;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_kf + s, 1);
            mbar_init(b_vf + s, 1);
            mbar_init(b_sf + s, 1);
            mbar_init(b_pf + s, 128);
            mbar_init(b_od + s, 1);
            mbar_init(b_ke + s, 1);
            mbar_init(b_ve + s, 1);
        }
        mbar_init(b_fin, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == kFwdProdWarp) {
        // chunk list: (KV row start within the batch entry, valid keys);
        // counts above idx_cap and tile ids outside [0, nKV) (invalid input,
        // reported by vsa_check_inputs) are clamped or skipped here
        const int cnt = clampi(a.q_cnt[qrow], 0, a.cap);
        const int *idx = a.q_idx + qrow * a.cap;
        const int per = p.tile_kv >> 7;
        int total = 0;
        for (int n0 = 0; n0 < cnt; n0 += 32) {
            const int n = n0 + lane;
            int j = 0, kvv = 0, nc = 0, bits = -1;
            if (n < cnt) {
                j = idx[n];
                kvv = (j >= 0 && j < p.nKV) ? kv_valid(p, b, j) : 0;
                nc = min(per, (kvv + 127) >> 7);
                if (a.q_sub) bits = a.q_sub[qrow * a.cap + n];
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
                    s_csub[pos] = bits;
                }
            }
            total += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) *s_nchunk = min(total, kMaxChunks);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *s_tmem;
    const int N = *s_nchunk;
    const bool bf16 = (p.dtype == T_BF16);
    int issued_q = 0, issued_k[2] = {0, 0}, issued_v[2] = {0, 0}, mma_started = 0;

    if (warp == kFwdProdWarp && lane == 0 && N > 0) {
        // ---------------------------------------------------- TMA producer
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        mbar_expect_tx(b_q, has_b ? 2 * kTile : kTile);
        for (int g = 0; g < (has_b ? 2 : 1); ++g) {
            tma_load_4d(sQ + g * kTile, &tq, b_q, 0, qbase + g * 128, h, bc);
            tma_load_4d(sQ + g * kTile + kBox, &tq, b_q, 64, qbase + g * 128, h, bc);
        }
        issued_q = 1;
        for (int c = 0; c < N; ++c) {
            const int s = c & 1;
            // stage s is free once the MMAs reading K(c-2) / V(c-2) are done;
            // each release barrier completes once per use of its stage, so
            // the producer can never be two phases behind it
            if (c >= 2 && !mbar_wait(b_ke + s, ((c >> 1) - 1) & 1, s_abort, a.err, kSiteProd)) break;
            const int kr = kvb + s_crow[c];
            mbar_expect_tx(b_kf + s, kTile);
            tma_load_4d(sK + s * kTile, &tk, b_kf + s, 0, kr, hk, bc);
            tma_load_4d(sK + s * kTile + kBox, &tk, b_kf + s, 64, kr, hk, bc);
            issued_k[s]++;
            if (c >= 2 && !mbar_wait(b_ve + s, ((c >> 1) - 1) & 1, s_abort, a.err, kSiteProd)) break;
            mbar_expect_tx(b_vf + s, kTile);
            tma_load_4d(sV + s * kTile, &tv, b_vf + s, 0, kr, hk, bc);
            tma_load_4d(sV + s * kTile + kBox, &tv, b_vf + s, 64, kr, hk, bc);
            issued_v[s]++;
        }
    } else if (warp == kFwdMmaWarp && N > 0) {
        // ------------------------------------- MMA issuer (whole warp, lane 0 issues)
        const uint32_t idS = idesc_f16(bf16, 128, 128, false, false);
        const uint32_t idO = idesc_f16(bf16, 128, 128, false, true);
        const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);
        const uint32_t tS[2] = {tbase, tbase + 128}, tO[2] = {tbase + 256, tbase + 384};
        bool ok = mbar_wait_warp(b_q, 0, s_abort, a.err, kSiteMma);
        for (int c = 0; ok && c < N; ++c) {
            const int s = c & 1, sp = (c - 1) & 1;
            if (!(ok = mbar_wait_warp(b_kf + s, (c >> 1) & 1, s_abort, a.err, kSiteMma))) break;
            tc_fence_after();
            issue_qk(tS[0], aQ, aK + s * kTile, idS);  // S_A(c); P_A(c-1) was consumed by PV_A(c-1)
            mma_commit_w(b_sf + 0);
            mma_started = 1;
            if (has_b) {
                if (c > 0) {
                    if (!(ok = mbar_wait_warp(b_pf + 1, (c - 1) & 1, s_abort, a.err, kSiteMma))) break;
                    tc_fence_after();
                    issue_pv(tO[1], tS[1], aV + sp * kTile, idO, c - 1 > 0);  // O_B += P_B(c-1) V_(c-1)
                    mma_commit_w(b_ve + sp);  // V_(c-1) read by both groups
                }
                issue_qk(tS[1], aQ + kTile, aK + s * kTile, idS);  // S_B(c)
                mma_commit_w(b_sf + 1);
            }
            mma_commit_w(b_ke + s);  // K_c is read by the S MMAs only
            if (!(ok = mbar_wait_warp(b_pf + 0, c & 1, s_abort, a.err, kSiteMma))) break;
            if (!(ok = mbar_wait_warp(b_vf + s, (c >> 1) & 1, s_abort, a.err, kSiteMma))) break;
            tc_fence_after();
            issue_pv(tO[0], tS[0], aV + s * kTile, idO, c > 0);  // O_A += P_A(c) V_c
            if (c == N - 1) mma_commit_w(b_od + 0);  // O_A final (S_A(c+1) would signal it otherwise)
            if (!has_b) mma_commit_w(b_ve + s);
        }
        if (ok && has_b) {
            const int sp = (N - 1) & 1;
            if (mbar_wait_warp(b_pf + 1, (N - 1) & 1, s_abort, a.err, kSiteMma)) {
                tc_fence_after();
                issue_pv(tO[1], tS[1], aV + sp * kTile, idO, N - 1 > 0);
                mma_commit_w(b_od + 1);
                mma_commit_w(b_ve + sp);
            }
        }
    } else if (warp < 8 && (warp < 4 || has_b)) {
        // -------------------------------------------- softmax + epilogue
        const int g = warp >> 2, lg = warp & 3;
        const int r = lg * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(lg * 32) << 16);
        const uint32_t cS = g * 128, cO = 256 + g * 128;
        const float sl2 = p.scale * kLog2e;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int c = 0; c < N; ++c) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_sf + g, c & 1, s_abort, a.err, kSiteSoft));
            if (!ok) break;
            tc_fence_after();
            int valid = s_cval[c];
            // query blocks: a row whose block did not select this tile sees no key of it
            if (a.q_sub && !((s_csub[c] >> ((g * 128 + r) / a.block_q)) & 1)) valid = 0;
            // The whole row of S (128 scores) comes into registers with one
            // wait. Probabilities are exp2(scale log2e s - m_ref) against the
            // row's running reference m_ref, packed into the first 64 columns
            // of the S buffer. Once the row has a reference, the chunk goes
            // straight to the exponentials: fp32 and the 16-bit P keep their
            // relative precision at any magnitude, so m_ref only has to keep
            // P finite, and a row sum within kSumLimit bounds every element.
            // The first chunk, and a chunk whose sum passes the limit, take
            // the row max first (the scale is positive, so on raw scores) and
            // move m_ref to it when it is more than 2^8 above (rescaling l and
            // O in TMEM), then redo the exponentials.
            uint32_t sr[128];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tl + cS + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + q4 * 32));
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(sr + q4 * 32));
            if (valid < 128) {
#pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
            }
            float ls = 0.f, alpha = 1.f;
            bool slow = m_ref == -INFINITY;
            if (!__any_sync(0xffffffffu, slow)) {
                ls = exp_row<T>(sr, m_ref, sl2, tl + cS);
                slow = !(ls <= SumLimit<T>::value);  // also true for inf / nan
                if (__any_sync(0xffffffffu, slow)) tmem_wait_st();  // the redo below overwrites these stores
            }
            if (__any_sync(0xffffffffu, slow)) {
                float mx;
                {
                    float u[43], v[15], w5[5];
#pragma unroll
                    for (int k = 0; k < 42; ++k)
                        u[k] = fmax3(__uint_as_float(sr[3 * k]), __uint_as_float(sr[3 * k + 1]),
                                     __uint_as_float(sr[3 * k + 2]));
                    u[42] = fmaxf(__uint_as_float(sr[126]), __uint_as_float(sr[127]));
#pragma unroll
                    for (int k = 0; k < 14; ++k) v[k] = fmax3(u[3 * k], u[3 * k + 1], u[3 * k + 2]);
                    v[14] = u[42];
#pragma unroll
                    for (int k = 0; k < 5; ++k) w5[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
                    mx = fmaxf(fmax3(w5[0], w5[1], w5[2]), fmaxf(w5[3], w5[4])) * sl2;
                }
                if (mx > m_ref + 8.f) {
                    alpha = ex2(m_ref - mx);  // 0 on the first chunk
                    m_ref = mx;
                }
                // (a row that has seen no key yet keeps m_ref = -inf; its
                // scores are all -inf and must give P = 0, not inf - inf)
                ls = exp_row<T>(sr, m_ref == -INFINITY ? 0.f : m_ref, sl2, tl + cS);
            }
            const bool resc = alpha != 1.f;
            l = l * alpha + ls;
            // O_g += P_g(c-1) V_(c-1) was issued before S_g(c), which is done
            if (c > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t o[32];
                    tmem_ld32(tl + cO + q4 * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(tl + cO + q4 * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_pf + g);
        }
        if (ok && N > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_od + g, 0, s_abort, a.err, kSiteEpi));  // committed once
            if (ok) tc_fence_after();
        }
        const bool have = ok && N > 0;                 // warp-uniform: TMEM holds O
        const bool row_has = have && l > 0.f;           // l = 0: the row saw no key (O = 0, LSE = -inf)
        const float inv_l = row_has ? 1.f / l : 0.f;
        const float lse_v = row_has ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        const bool row_ok = r < nrows[g];
        const int row = i * p.tile_q + g * 128 + r;  // within the batch entry
        const long long ro = tok_off(p, true, b, row, h);
        T *osp = a.o_sparse ? reinterpret_cast<T *>(a.o_sparse) + ro : nullptr;
        T *out = reinterpret_cast<T *>(a.out) + ro;
        const T *gt = a.gate ? reinterpret_cast<const T *>(a.gate) + ro : nullptr;
        const float *cc = a.gate ? a.c + qrow * 128 : nullptr;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tl + cO + q4 * 32, o);
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
        if (row_ok && a.lse) a.lse[lse_off(p, b, h, row)] = lse_v;
    }

    // ------------------------------------------------------------ teardown
    if (*s_abort) {
        // Drain what this CTA started before leaving: outstanding TMA copies
        // (producer) and MMAs (issuer), each with a bounded wait.
        int never = 0;
        if (warp == kFwdProdWarp && lane == 0) {
            if (issued_q) mbar_wait(b_q, 0, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < 2; ++s) {
                if (issued_k[s]) mbar_wait(b_kf + s, (issued_k[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
                if (issued_v[s]) mbar_wait(b_vf + s, (issued_v[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
            }
        }
    }
    if (warp == kFwdMmaWarp && mma_started && __any_sync(0xffffffffu, *s_abort != 0)) {
        // the MMAs this warp issued finish before TMEM is released
        int never = 0;
        mma_commit_w(b_fin);
        __all_sync(0xffffffffu, mbar_wait(b_fin, 0, &never, nullptr, 0, 200000000ull));
    }
    tc_fence_before();
    __syncthreads();  // every wait on this tile's barriers is over
    if (threadIdx.x == 0)
        for (int x = 0; x < kFwdBars; ++x) mbar_inval(bars + x);
}

// One tile per CTA; in the redo launch (redo_only) a CTA takes kRedoGroup
// consecutive query tiles of one head and computes those marked in redo,
// one after the other (a CTA none of whose tiles is marked leaves at once,
// so the launch costs little when nothing is marked).
template <typename T>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
          const __grid_constant__ CUtensorMap tv, const Prob p, const FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    const int h = blockIdx.y, b = blockIdx.z;
    const long long row0 = ((long long)b * p.Hq + h) * p.nQ;
    const int i0 = a.redo_only ? (int)blockIdx.x * kRedoGroup : (int)blockIdx.x;
    const int ntiles = a.redo_only ? min(kRedoGroup, p.nQ - i0) : 1;
    if (a.redo_only) {
        bool any = false;
        for (int x = 0; x < ntiles; ++x) any = any || a.redo[row0 + i0 + x] != 0;
        if (!any) return;
    }
    if ((smem_addr(sm) & 1023u) != 0) {  // the swizzled operand tiles need 1024-byte alignment
        if (threadIdx.x == 0) set_error(a.err, 0x1FF);
        return;
    }
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kOffCtl + kFwdBars * 8);
    const int warp = threadIdx.x >> 5;
    if (warp == kFwdMmaWarp) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    for (int x = 0; x < ntiles; ++x) {
        if (a.redo_only && !a.redo[row0 + i0 + x]) continue;
        fwd_tile<T>(tq, tk, tv, p, a, sm, i0 + x, h, b);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kFwdMmaWarp) {
        tc_fence_after();
        tmem_dealloc(*s_tmem, 512);
    }
}

// ------------------------------------------------ forward on a CTA pair
// 256-token query tiles without query-block masks: a cluster of two CTAs
// takes one tile, CTA r (its cluster rank) the 128-row group r. The even
// CTA issues M = 256 MMAs (tcgen05 cta_group::2) for both: each CTA holds
// its own 128 rows of Q, S, P and O, keys [64r, 64r + 64) of each 128-key
// K chunk and head dims [64r, 64r + 64) of each V chunk, so a chunk costs
// each SM 32 KB of loads for its 128 rows and six K/V stages fit beside Q.
// TMEM holds three S buffers and O, so S(c+3) is issued right after
// O += P(c) V(c). The loads of both CTAs complete on the even CTA's
// barriers; every MMA commit arrives in both CTAs.
// Softmax: the two warps of a TMEM lane quarter (32 rows) take alternate
// chunks, each whole rows, so one warp's waits overlap the other's
// exponentials. Every row's reference is its max over chunk 0, kept for
// all chunks: fp32 and the 16-bit P keep their relative precision at any
// magnitude, so nothing is rescaled. A chunk whose row sum passes
// SumLimit (an element that the 16-bit P cannot hold) marks the tile in
// `redo`; the single-CTA kernel, which moves its reference, recomputes
// exactly those tiles right after. Each chunk's P is handed to the O += P V
// issuer in two halves (keys 0..63, then 64..127), so the first four
// K = 16 steps run while the softmax finishes the row. In padded layouts
// the epilogue stages its rows in shared memory in the TMA box layout and
// writes them with box stores when O is the only output, or when gated:
// out in the Q buffer and O (the sparse output) in the first two K stages.
// The gated instantiation (kGated) copies the gate's rows into the Q
// buffer as soon as the last S MMA has read Q, while the last chunks'
// softmax and O += P V still run, and its epilogue turns them into
// out = O + gate * c in place; the ungated one has none of this code.
// Warp roles (each CTA): warps 0-7 softmax (warp w: TMEM lanes 32 (w % 4),
// chunks of parity w / 4, and in the epilogue O columns [64 (w / 4), +64)),
// warp 8 loads, warp 9 owns TMEM and (even CTA) issues the S MMAs, warp 10
// (even CTA) issues the O += P V MMAs.
// TMEM columns: S buffers [0,128), [128,256), [256,384) (P packed into the
// first 64 columns of its S buffer), O [384,512).
constexpr int kF2Stages = 6;
constexpr int kF2Q = 32 * 1024;   // Q of the CTA's 128 rows: two 64-column boxes of 128 rows
constexpr int kF2KH = 16 * 1024;  // half a K chunk: 64 keys x 128 dims, two 64-column boxes of 64 rows
constexpr int kF2VH = 16 * 1024;  // half a V chunk: 128 keys x 64 dims, one box
constexpr int kF2OffK = kF2Q, kF2OffV = kF2OffK + kF2Stages * kF2KH, kF2OffCtl = kF2OffV + kF2Stages * kF2VH;
constexpr size_t kF2Smem = kF2OffCtl + 2560;
constexpr int kF2Threads = 352, kF2ProdWarp = 8, kF2MmaWarp = 9, kF2PvWarp = 10;
enum : unsigned { kSite2Prod = 0x111, kSite2Mma = 0x112, kSite2Soft = 0x113, kSite2Epi = 0x114 };

// S = Q K_half^T for one chunk on the pair: A = the CTA's Q (boxes 16 KB
// apart), B = its 64 keys (boxes 8 KB apart); 8 MMAs of K = 16.
__device__ __forceinline__ void issue_qk2(uint32_t d, uint32_t aQ, uint32_t aK, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma2_ss_w(d, sdesc_sw128(aQ + (kk >> 2) * (kF2Q / 2) + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(aK + (kk >> 2) * (kF2KH / 2) + (kk & 3) * 32, 16, 1024), idesc, kk > 0);
}
// O += P V_half on the pair: A = P in TMEM (128 keys packed in the S
// buffer's first 64 columns, 8 per K = 16 step), B = the CTA's 64 head
// dims of the chunk's 128 keys, read MN-major (8-key groups 1 KB apart);
// K = 16 steps [K0, K1).
template <int K0, int K1>
__device__ __forceinline__ void issue_pv2(uint32_t d, uint32_t p_tmem, uint32_t aV, uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = K0; kk < K1; ++kk)
        mma2_ts_w(d, p_tmem + kk * 8, sdesc_sw128(aV + kk * 2048, kF2VH, 1024), idesc, (acc || kk > 0) ? 1u : 0u);
}

template <typename T, bool kGated>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kF2Threads, 1)
    k_fwd2(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
           const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tout,
           const __grid_constant__ CUtensorMap tgate, const __grid_constant__ CUtensorMap tosp, const Prob p,
           const FwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x >> 1, h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    // both CTAs of the pair take the same early exits, before any cluster interaction
    const int tile_rows = p.layout == L_TND ? clampi(seq_len(p, true, b) - i * p.tile_q, 0, p.tile_q) : p.tile_q;
    if (tile_rows == 0) {  // the whole tile lies outside its sequence
        if (threadIdx.x == 0 && rank == 0 && a.redo) a.redo[((long long)b * p.Hq + h) * p.nQ + i] = 0;
        return;
    }
    if ((smem_addr(sm) & 1023u) != 0) {  // the swizzled operand tiles need 1024-byte alignment
        if (threadIdx.x == 0) set_error(a.err, 0x1FE);
        return;
    }
    const int nrows = clampi(tile_rows - (int)rank * 128, 0, 128);
    const bool leader = rank == 0;
    uint8_t *sQ = sm, *sK = sm + kF2OffK, *sV = sm + kF2OffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kF2OffCtl);
    uint64_t *b_q = bars, *b_kv = bars + 1, *b_free = b_kv + kF2Stages, *b_s = b_free + kF2Stages;
    uint64_t *b_p = b_s + 3, *b_o = b_p + 3, *b_fin = b_o + 1, *b_mref = b_fin + 2;
    uint64_t *b_pvd = b_mref + 1;  // (even CTA) O += P V of buffer x's chunk done: x may take S again
    uint64_t *b_plo = b_pvd + 3;   // (even CTA) P of buffer x's first 64 keys stored, in both CTAs
    uint64_t *b_qd = b_plo + 3;    // the last S MMA has read Q (both CTAs)
    uint64_t *b_g = b_qd + 1;      // this CTA's gate rows have landed in the Q buffer
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(sm + kF2OffCtl + 256);  // after 31 barriers (248 bytes)
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nchunk = reinterpret_cast<int *>(s_tmem + 2);
    volatile int *s_over = reinterpret_cast<volatile int *>(s_tmem + 3);       // a chunk passed SumLimit here
    volatile int *s_over_peer = reinterpret_cast<volatile int *>(s_tmem + 4);  // the odd CTA's flag (even CTA)
    float *s_mref = reinterpret_cast<float *>(sm + kF2OffCtl + 512);           // [128] rows' references
    float *s_lsum = reinterpret_cast<float *>(sm + kF2OffCtl + 1024);          // [2][128] row-sum parts

    const int qbase = (p.layout == L_TND ? seq_start(p, true, b) : 0) + i * p.tile_q + (int)rank * 128;
    const int kvb = (p.layout == L_TND ? seq_start(p, false, b) : 0);
    const int bc = (p.layout == L_TND ? 0 : b);
    const long long qrow = ((long long)b * p.Hq + h) * p.nQ + i;
    const int cnt = clampi(a.q_cnt[qrow], 0, a.cap);  // counts past idx_cap are invalid input
    // the producer reads the row's first 32 entries without waiting for
    // their count (a row holds idx_cap entries), so the two reads overlap
    const int jfirst = (warp == kF2ProdWarp && lane < a.cap) ? a.q_idx[qrow * a.cap + lane] : -1;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < kF2Stages; ++s) {
            mbar_init(b_kv + s, 1);
            mbar_init(b_free + s, 1);
        }
        for (int x = 0; x < 3; ++x) {
            mbar_init(b_s + x, 1);
            mbar_init(b_p + x, 8);  // the 4 softmax warps of the chunk's parity in each CTA
        }
        mbar_init(b_o, 1);
        mbar_init(b_fin, 1);
        mbar_init(b_fin + 1, 1);
        mbar_init(b_mref, 4);  // the four warps that take chunk 0
        for (int x = 0; x < 3; ++x) mbar_init(b_pvd + x, 1);
        for (int x = 0; x < 3; ++x) mbar_init(b_plo + x, 8);  // as b_p
        if constexpr (kGated) {
            mbar_init(b_qd, 1);
            mbar_init(b_g, 1);
        }
        *s_abort = 0;
        *s_over = 0;
        *s_over_peer = 0;
        fence_mbar_init();
    }
    // The producer reads the selection before the cluster sync: the chunk
    // count every role needs, and the first window of its own walk, so
    // that Q and the first K/V chunk are requested right after the sync.
    ChunkWin pcw{};
    if (warp == kF2ProdWarp) {
        // number of 128-key chunks with valid keys (tile ids outside [0, nKV) skipped, as the walk does)
        const int *idx = a.q_idx + qrow * a.cap;
        const int per = p.tile_kv >> 7;
        int total = 0;
        for (int n = lane; n < cnt; n += 32) {
            const int j = n < 32 ? jfirst : idx[n];
            total += (j >= 0 && j < p.nKV) ? min(per, (kv_valid(p, b, j) + 127) >> 7) : 0;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
        if (lane == 0) *s_nchunk = total;
        pcw = win_begin(p, b, idx, nullptr, cnt, lane);
    } else if (warp == kF2MmaWarp) {
        tmem_alloc2(s_tmem, 512);
        tmem_relinquish2();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated in both
    tc_fence_after();
    const uint32_t tbase = *s_tmem;
    const int N = *s_nchunk;
    const bool bf16 = (p.dtype == T_BF16);
    int issued_kv = 0, mma_started = 0;

    if (warp == kF2ProdWarp && N > 0) {
        // ------------------------------------------------------ producer (whole warp walks the chunks)
        ChunkWin &cw = pcw;
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            const uint32_t cq = cluster_addr(smem_addr(b_q), 0);
            if (leader) mbar_expect_tx(b_q, 2 * kF2Q);
            tma_load_4d_pair(sQ, &tq, cq, 0, qbase, h, bc);
            tma_load_4d_pair(sQ + kF2Q / 2, &tq, cq, 64, qbase, h, bc);
        }
        for (int c = 0; c < N; ++c) {
            int crow = 0, cval = 0, cbits = -1;
            if (!win_chunk(p, b, cw, c, lane, crow, cval, cbits)) break;
            const int st = c % kF2Stages;
            // the stage is free once O += P V of its previous chunk is done (in both CTAs)
            if (c >= kF2Stages &&
                !mbar_wait_warp(b_free + st, ((c / kF2Stages) - 1) & 1, s_abort, a.err, kSite2Prod))
                break;
            if (lane == 0) {
                // one barrier round per chunk for K and V together (both CTAs' halves)
                const uint32_t ckv = cluster_addr(smem_addr(b_kv + st), 0);
                if (leader) mbar_expect_tx(b_kv + st, 2 * (kF2KH + kF2VH));
                const int kr = kvb + crow;
                uint8_t *dK = sK + st * kF2KH, *dV = sV + st * kF2VH;
                tma_load_4d_pair(dK, &tk, ckv, 0, kr + (int)rank * 64, hk, bc);
                tma_load_4d_pair(dK + kF2KH / 2, &tk, ckv, 64, kr + (int)rank * 64, hk, bc);
                tma_load_4d_pair(dV, &tv, ckv, (int)rank * 64, kr, hk, bc);
            }
            issued_kv = c + 1;
        }
        if constexpr (kGated) {
            // the gate's rows into the Q buffer once the last S MMA has read it
            if (p.layout != L_TND && lane == 0 && issued_kv == N && mbar_wait(b_qd, 0, s_abort, a.err, kSite2Prod)) {
                tma_prefetch_desc(&tgate);
                mbar_expect_tx(b_g, kF2Q);
                tma_load_4d(sQ, &tgate, b_g, 0, qbase, h, bc);
                tma_load_4d(sQ + kF2Q / 2, &tgate, b_g, 64, qbase, h, bc);
            }
        }
    } else if (warp == kF2MmaWarp && leader && N > 0) {
        // --------------------------- S issuer of the pair (whole warp, one lane issues)
        // S(c) goes into buffer c % 3 once K(c) has landed and O += P V has
        // read the chunk three back from that buffer.
        const uint32_t idS = idesc_f16(bf16, 256, 128, false, false);
        const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK);
        bool ok = mbar_wait_warp(b_q, 0, s_abort, a.err, kSite2Mma);
        for (int c = 0; ok && c < N; ++c) {
            const int st = c % kF2Stages, x = c % 3;
            if (c >= 3 && !(ok = mbar_wait_warp(b_pvd + x, ((c / 3) - 1) & 1, s_abort, a.err, kSite2Mma))) break;
            if (!(ok = mbar_wait_warp(b_kv + st, (c / kF2Stages) & 1, s_abort, a.err, kSite2Mma))) break;
            tc_fence_after();
            issue_qk2(tbase + x * 128, aQ, aK + st * kF2KH, idS);
            mma2_commit_mc_w(b_s + x, 3);
            mma_started = 1;
        }
        if constexpr (kGated) {
            if (ok && p.layout != L_TND) mma2_commit_mc_w(b_qd, 3);  // Q read by every S MMA, in both CTAs
        }
    } else if (warp == kF2PvWarp && leader && N > 0) {
        // ------------------------ PV issuer of the pair (whole warp, one lane issues)
        // Its waits for P overlap the S issuer's MMAs and the other way round.
        // S(c) completed before the softmax could write P(c), so once
        // O += P(c) V(c) is done both K(c) and V(c) are read.
        const uint32_t idO = idesc_f16(bf16, 256, 128, false, true);
        const uint32_t aV = smem_addr(sV);
        const uint32_t tO = tbase + 384;
        bool ok = true;
        for (int c = 0; ok && c < N; ++c) {
            const int st = c % kF2Stages, x = c % 3;
            // O += P(c) V(c) in two halves: keys 0..63 as soon as their P
            // is stored, keys 64..127 once the softmax has finished the row
            if (!(ok = mbar_wait_warp(b_plo + x, (c / 3) & 1, s_abort, a.err, kSite2Mma))) break;
            tc_fence_after();
            issue_pv2<0, 4>(tO, tbase + x * 128, aV + st * kF2VH, idO, c > 0);
            mma_started = 1;
            if (!(ok = mbar_wait_warp(b_p + x, (c / 3) & 1, s_abort, a.err, kSite2Mma))) break;
            tc_fence_after();
            issue_pv2<4, 8>(tO, tbase + x * 128, aV + st * kF2VH, idO, true);
            mma2_commit_mc_w(b_free + st, 3);  // K(c), V(c) read, in both CTAs
            mma2_commit_mc_w(b_pvd + x, 1);    // P(c) read: buffer x may take S(c + 3)
        }
        if (ok) mma2_commit_mc_w(b_o, 3);
    } else if (warp < 8) {
        // ------------------------------------------------------ softmax + epilogue
        const int lg = warp & 3, grp = warp >> 2;  // lane quarter, parity of the chunks this warp takes
        const int r = lg * 32 + lane;             // row within the CTA's group
        const uint32_t tl = tbase + ((uint32_t)(lg * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        float m_ref = -INFINITY, l = 0.f;  // l: the part of the row sum from this warp's chunks
        bool ok = true, over = false;
        ChunkWin cw = win_begin(p, b, a.q_idx + qrow * a.cap, nullptr, cnt, lane);
        const uint32_t cp0 = cluster_addr(smem_addr(b_p), 0);
        const uint32_t cplo = cluster_addr(smem_addr(b_plo), 0);
        for (int c = grp; c < N; c += 2) {
            const int x = c % 3;
            int crow = 0, valid = 0, cbits = -1;
            win_chunk(p, b, cw, c, lane, crow, valid, cbits);
            if (!(ok = mbar_wait_warp(b_s + x, (c / 3) & 1, s_abort, a.err, kSite2Soft))) break;
            tc_fence_after();
            uint32_t sr[128];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_ld32(tl + x * 128 + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + q4 * 32));
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(sr + q4 * 32));
            if (valid < 128) {
#pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
            }
            if (c == 0) {
                // the row's reference: its max over the first chunk (every
                // chunk holds at least one valid key, so it is finite)
                float u[43], v[15], w5[5];
#pragma unroll
                for (int k = 0; k < 42; ++k)
                    u[k] = fmax3(__uint_as_float(sr[3 * k]), __uint_as_float(sr[3 * k + 1]),
                                 __uint_as_float(sr[3 * k + 2]));
                u[42] = fmaxf(__uint_as_float(sr[126]), __uint_as_float(sr[127]));
#pragma unroll
                for (int k = 0; k < 14; ++k) v[k] = fmax3(u[3 * k], u[3 * k + 1], u[3 * k + 2]);
                v[14] = u[42];
#pragma unroll
                for (int k = 0; k < 5; ++k) w5[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
                m_ref = fmaxf(fmax3(w5[0], w5[1], w5[2]), fmaxf(w5[3], w5[4])) * sl2;
                s_mref[r] = m_ref;
                __syncwarp();
                if (lane == 0) mbar_arrive(b_mref);
            } else if (m_ref == -INFINITY) {  // this warp's first chunk: take chunk 0's reference
                if (!(ok = mbar_wait_warp(b_mref, 0, s_abort, a.err, kSite2Soft))) break;
                m_ref = s_mref[r];
            }
            // P of keys 0..63 first, handed over before keys 64..127
            float ls = exp_row<T, 0, 2>(sr, m_ref, sl2, tl + x * 128);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(cplo + 8u * x);
            ls += exp_row<T, 2, 4>(sr, m_ref, sl2, tl + x * 128);
            over = over || !(ls <= SumLimit<T>::value);
            l += ls;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(cp0 + 8u * x);
        }
        if (__any_sync(0xffffffffu, over) && lane == 0) *s_over = 1;
        if (ok && N > 0) {
            ok = mbar_wait_warp(b_o, 0, s_abort, a.err, kSite2Epi);
            if (ok) tc_fence_after();
        }
        // gated padded layouts: the gate's rows come by TMA once Q is no
        // longer read (with no chunk no MMA runs and the gate is read directly)
        const bool gate_tma = kGated && p.layout != L_TND && N > 0;
        if (ok && gate_tma) ok = mbar_wait_warp(b_g, 0, s_abort, a.err, kSite2Epi);
        // the row sum: both warps' parts (every softmax warp comes here once)
        s_lsum[grp * 128 + r] = l;
        named_sync(1, 256);
        const float lt = s_lsum[r] + s_lsum[128 + r];
        // the O columns of this warp: [64 grp, 64 grp + 64)
        const int ch = grp;
        const bool have = ok && N > 0;                  // warp-uniform: TMEM holds O
        const bool row_has = have && lt > 0.f;          // lt = 0: the row saw no key (O = 0, LSE = -inf)
        const float inv_l = row_has ? 1.f / lt : 0.f;
        const float lse_v = row_has ? (m_ref + __log2f(lt)) * kLn2 : -INFINITY;
        const bool row_ok = r < nrows;
        const int row = i * p.tile_q + (int)rank * 128 + r;  // within the batch entry
        const long long ro = tok_off(p, true, b, row, h) + ch * 64;
        T *osp = a.o_sparse ? reinterpret_cast<T *>(a.o_sparse) + ro : nullptr;
        T *out = reinterpret_cast<T *>(a.out) + ro;
        const T *gt = a.gate ? reinterpret_cast<const T *>(a.gate) + ro : nullptr;
        const float *cc = a.gate ? a.c + qrow * 128 + ch * 64 : nullptr;
        // One output (no gate, O kept only as out), padded layout: the CTA's
        // 128 rows of O are staged in its Q buffer (free once the last S MMA
        // is done) in the TMA box layout and stored by two box copies.
        const bool staged = p.layout != L_TND && !a.gate && (!a.o_sparse || a.o_sparse == a.out);
        // Gated, padded layout: out = O + gate (*) c is staged in the Q
        // buffer (where the gate's rows are), O in the first two K stages
        // (free once O is complete), both in the TMA box layout.
        const bool gstaged = kGated && p.layout != L_TND;
        if constexpr (kGated) {
#pragma unroll 1
            for (int q2 = 0; q2 < 2; ++q2) {
                uint32_t o[32];
                if (have) {
                    tmem_ld32(tl + 384 + ch * 64 + q2 * 32, o);
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
                // columns 64 ch + 32 q2 .. +31: box ch, 16-byte chunks 4 q2 .. +3 of row r, 128-byte swizzle
                uint8_t *rq = sQ + ch * (kF2Q / 2) + r * 128, *rk = sK + ch * (kF2Q / 2) + r * 128;
                if (gstaged && osp) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *reinterpret_cast<uint4 *>(rk + (((q2 * 4 + u) ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
                if (osp && !gstaged) {
                    uint4 *dst = reinterpret_cast<uint4 *>(osp + q2 * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
                const uint4 *gsrc = reinterpret_cast<const uint4 *>(gt + q2 * 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 gv = gate_tma ? *reinterpret_cast<const uint4 *>(rq + (((q2 * 4 + u) ^ (r & 7)) << 4))
                                              : gsrc[u];
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float2 g2 = unpack2<T>(gw[t]);
                        const int e = q2 * 32 + u * 8 + t * 2;
                        w[u * 4 + t] = pack2<T>(vals[u * 8 + t * 2] + g2.x * cc[e],
                                                vals[u * 8 + t * 2 + 1] + g2.y * cc[e + 1]);
                    }
                }
                if (gstaged) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *reinterpret_cast<uint4 *>(rq + (((q2 * 4 + u) ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + q2 * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
            }
        } else {
#pragma unroll 1
            for (int q2 = 0; q2 < 2; ++q2) {
                uint32_t o[32];
                if (have) {
                    tmem_ld32(tl + 384 + ch * 64 + q2 * 32, o);
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
                if (osp && !staged) {
                    uint4 *dst = reinterpret_cast<uint4 *>(osp + q2 * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
                if (gt) {
                    const uint4 *gsrc = reinterpret_cast<const uint4 *>(gt + q2 * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 gv = gsrc[u];
                        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float2 g2 = unpack2<T>(gw[t]);
                            const int e = q2 * 32 + u * 8 + t * 2;
                            w[u * 4 + t] = pack2<T>(vals[u * 8 + t * 2] + g2.x * cc[e],
                                                    vals[u * 8 + t * 2 + 1] + g2.y * cc[e + 1]);
                        }
                    }
                }
                if (staged) {
                    // columns 64 ch + 32 q2 .. +31: box ch, 16-byte chunks 4 q2 .. +3 of row r, 128-byte swizzle
                    uint8_t *rowp = sQ + ch * (kF2Q / 2) + r * 128;
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        *reinterpret_cast<uint4 *>(rowp + (((q2 * 4 + u) ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                } else if (gt || out != osp) {
                    uint4 *dst = reinterpret_cast<uint4 *>(out + q2 * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
            }
        }
        if (row_ok && ch == 0 && a.lse) a.lse[lse_off(p, b, h, row)] = lse_v;
        if (gstaged || staged) {
            fence_proxy_async_smem();
            named_sync(1, 256);  // the 8 softmax warps have staged their rows
            if (warp == 0 && lane == 0 && !*s_abort) {
                tma_store_4d(&tout, sQ, 0, qbase, h, bc);
                tma_store_4d(&tout, sQ + kF2Q / 2, 64, qbase, h, bc);
                if (gstaged && a.o_sparse && a.o_sparse != a.out) {
                    tma_store_4d(&tosp, sK, 0, qbase, h, bc);
                    tma_store_4d(&tosp, sK + kF2Q / 2, 64, qbase, h, bc);
                }
                tma_store_commit();
                tma_store_wait_read();  // the stage is read before this CTA's shared memory goes
            }
        }
    }

    // ------------------------------------------------------------ teardown
    if (*s_abort) {
        // Loads of both CTAs complete on the even CTA's barriers, which a
        // half-fed phase never completes: give copies in flight time to land
        // before this CTA's shared memory can be released.
        if (warp == kF2ProdWarp && lane == 0 && issued_kv + 1 > 0) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 100000ull) {
            }
        }
        if ((warp == kF2MmaWarp || warp == kF2PvWarp) && mma_started) {
            // the MMAs this warp issued finish before TMEM is released
            int never = 0;
            uint64_t *bf = b_fin + (warp == kF2PvWarp ? 1 : 0);
            mma2_commit_mc_w(bf, 1);
            __all_sync(0xffffffffu, mbar_wait(bf, 0, &never, nullptr, 0, 200000000ull));
        }
    }
    // the odd CTA's overflow flag goes to the even CTA, which records the tile
    if (!leader && threadIdx.x == 0) {
        const uint32_t dst = cluster_addr(smem_addr(const_cast<int *>(s_over_peer)), 0);
        const int v = *s_over;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(dst), "r"(v) : "memory");
    }
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while the other may still touch its barriers or TMEM
    if (leader && threadIdx.x == 0 && a.redo) a.redo[qrow] = (*s_over || *s_over_peer) ? 1 : 0;
    if (warp == kF2MmaWarp) {
        tc_fence_after();
        tmem_dealloc2(tbase, 512);
    }
}

}  // namespace

cudaError_t launch_fwd(const Prob &p, const FwdArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_rows(&tq, p, true, a.q, p.Hq) || !make_tmap_rows(&tk, p, false, a.k, p.Hkv) ||
        !make_tmap_rows(&tv, p, false, a.v, p.Hkv))
        return cudaErrorInvalidValue;
    if (p.nQ == 0 || p.Hq == 0 || p.B == 0) return cudaSuccess;
    FwdArgs a1 = a;
    a1.redo_only = 0;
    if (p.tile_q == 256 && !a.q_sub && a.redo) {
        // a CTA pair per 256-token query tile; the tiles it marks in redo
        // are then recomputed by the single-CTA kernel below
        CUtensorMap tk2, tout, tgate, tosp;
        if (!make_tmap_rows(&tk2, p, false, a.k, p.Hkv, 64) || !make_tmap_rows(&tout, p, true, a.out, p.Hq))
            return cudaErrorInvalidValue;
        tgate = tout;  // read only when gated
        tosp = tout;   // written only when O is a separate tensor
        if ((a.gate && !make_tmap_rows(&tgate, p, true, a.gate, p.Hq)) ||
            (a.o_sparse && a.o_sparse != a.out && !make_tmap_rows(&tosp, p, true, a.o_sparse, p.Hq)))
            return cudaErrorInvalidValue;
        dim3 grid2(2 * p.nQ, p.Hq, p.B);
        // the gated instantiation adds the gate's copy and the staged sum;
        // the other one compiles without any of it
        const void *kern = p.dtype == T_BF16 ? (a.gate ? (const void *)k_fwd2<__nv_bfloat16, true>
                                                       : (const void *)k_fwd2<__nv_bfloat16, false>)
                                             : (a.gate ? (const void *)k_fwd2<__half, true>
                                                       : (const void *)k_fwd2<__half, false>);
        const cudaError_t ae = ensure_smem_limit(kern, (int)kF2Smem);
        if (ae != cudaSuccess) return ae;
        prof_begin("fwd_attn", s);
        if (p.dtype == T_BF16) {
            if (a.gate)
                k_fwd2<__nv_bfloat16, true><<<grid2, kF2Threads, kF2Smem, s>>>(tq, tk2, tv, tout, tgate, tosp, p, a1);
            else
                k_fwd2<__nv_bfloat16, false><<<grid2, kF2Threads, kF2Smem, s>>>(tq, tk2, tv, tout, tgate, tosp, p, a1);
        } else {
            if (a.gate)
                k_fwd2<__half, true><<<grid2, kF2Threads, kF2Smem, s>>>(tq, tk2, tv, tout, tgate, tosp, p, a1);
            else
                k_fwd2<__half, false><<<grid2, kF2Threads, kF2Smem, s>>>(tq, tk2, tv, tout, tgate, tosp, p, a1);
        }
        prof_end(s);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        a1.redo_only = 1;
    }
    dim3 grid(a1.redo_only ? (p.nQ + kRedoGroup - 1) / kRedoGroup : p.nQ, p.Hq, p.B);
    const cudaError_t ae = p.dtype == T_BF16 ? ensure_smem_limit((const void *)k_fwd<__nv_bfloat16>, (int)kFwdSmem)
                                             : ensure_smem_limit((const void *)k_fwd<__half>, (int)kFwdSmem);
    if (ae != cudaSuccess) return ae;
    prof_begin(a1.redo_only ? "fwd_redo" : "fwd_attn", s);
    if (p.dtype == T_BF16)
        k_fwd<__nv_bfloat16><<<grid, kFwdThreads, kFwdSmem, s>>>(tq, tk, tv, p, a1);
    else
        k_fwd<__half><<<grid, kFwdThreads, kFwdSmem, s>>>(tq, tk, tv, p, a1);
    prof_end(s);
    return cudaGetLastError();
}


}  // namespace vsa
