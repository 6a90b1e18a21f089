// bwd_kernels.cu -- block-sparse attention backward on tcgen05, plus the
// row-sum preprocess and the compression gate's gradient (the compression
// branch's own backward is in compress_kernels.cu).
//
// Pages: Ascend test_npu_block_sparse_attention_backward.py
// (_softmax_backward_np: dS = P (dP - rowsum(P dP)); the TND/GQA backward
// golden: dQ = dS K, dK += dS^T Q, dV += P^T dO, summed over the GQA group);
// FastVideo block_sparse_attn_cute_fwd.py (the backward is KV-owned over
// the transposed index; _CuteAttentionQ128.backward recomputes P from the
// saved LSE with softmax_scale = D^-0.5).
//
// rowsum(P dP) equals Dvec = rowsum(dO * O), computed once per query row
// by k_bwd_prep. The KV-owned pass k_dkdv and the Q-owned pass k_dq each
// recompute S and dP on the tensor core, so neither needs atomics and every
// output element is written by exactly one CTA. In padded layouts both
// write their rows through shared memory (the Q tiles, free by then) with
// TMA box stores.
#include <climits>
#include <type_traits>

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
constexpr int kDqThreads = 384, kDqMmaWarp = 10, kDqPMmaWarp = 11;  // dQ: three MMA-issuing warps
constexpr int kDkThreads = 352, kDkMma2Warp = 10;  // dK/dV: a second MMA-issuing warp
constexpr int kProdWarp = 8, kMmaWarp = 9;

// ------------------------------------------------------------------ prep
// Per query slot w of the padded tile layout [B, Hq, nQ * tile_q]:
// nlse2[w] = -LSE * log2(e) and ndvec[w] = -sum_d dO_d O_d (minus
// rowsum(P dP) of the softmax backward); both are stored negated so the
// consumers add them. Slots that are not query rows (past a varlen
// sequence's end) get nlse2 = -inf and ndvec = 0, so P = 0 there.
// HBM-bound streaming: a task is 64 consecutive slots of one (b, h). Two
// producer warps (one lane each) stream the tasks' dO and O rows ([64 x
// 128] 16-bit tiles, two 64-column TMA boxes each, 128-byte swizzle) into
// a ring of kPrepStages shared-memory stages, alternating stages between
// them: a producer completes about one barrier round per ~900 cycles
// whatever the ring depth, so the bytes per round (32 KB) and the number
// of producers set the rate an SM can pull. Three consumer warps take the
// tasks in turn, each lane two rows (lane and lane + 32), so a row's sum
// stays in its lane and the LSE read and both writes are coalesced
// 128-byte accesses. Tasks are numbered in memory order of dO and O
// (heads of a token adjacent in BSHD and TND, tokens of a head in BHSD)
// and dealt to the CTAs round robin, so the CTAs in flight read
// neighbouring memory.
constexpr int kPrepRows = 64;                     // slots per task
constexpr int kPrepStages = 6;
constexpr int kPrepBox = kPrepRows * 128;         // one 64-column box of 64 rows (bytes)
constexpr int kPrepStage = 4 * kPrepBox;          // dO and O, two boxes each
constexpr int kPrepConsumers = 3, kPrepProducers = 2;
constexpr int kPrepThreads = 32 * (kPrepConsumers + kPrepProducers);
constexpr size_t kPrepSmem = (size_t)kPrepStages * kPrepStage + 256;
// A thread that takes every n-th task meets a stage again after
// lcm(n, kPrepStages) tasks; that must be exactly one barrier phase later
// (kPrepStages tasks), or its parity wait could pass on an older phase.
static_assert(kPrepStages % kPrepProducers == 0, "each producer returns to a stage one phase later");
static_assert(kPrepStages % kPrepConsumers == 0, "each consumer returns to a stage one phase later");
enum : unsigned { kSitePrepProd = 0x401, kSitePrepCons = 0x402 };

__device__ __forceinline__ void prep_task(const Prob &p, int task, int groups, int &b, int &h, int &s0) {
    int g;
    if (p.layout == L_BHSD) {
        g = task % groups;
        const int bh = task / groups;
        h = bh % p.Hq;
        b = bh / p.Hq;
    } else {
        h = task % p.Hq;
        const int bg = task / p.Hq;
        g = bg % groups;
        b = bg / groups;
    }
    s0 = g * kPrepRows;
}

template <typename T>
__device__ __forceinline__ float prep_row_dot(const uint8_t *base, uint32_t r) {
    float acc = 0.f;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t off = hf * kPrepBox + sw128_off(r, u);
            const uint4 x = *reinterpret_cast<const uint4 *>(base + off);
            const uint4 y = *reinterpret_cast<const uint4 *>(base + 2 * kPrepBox + off);
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a2 = unpack2<T>(xw[e]), c2 = unpack2<T>(yw[e]);
                acc = fmaf(a2.x, c2.x, acc);
                acc = fmaf(a2.y, c2.y, acc);
            }
        }
    }
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(kPrepThreads, 1)
    k_bwd_prep(const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap to, const Prob p,
               const float *__restrict__ lse, float *__restrict__ nlse2, float *__restrict__ ndvec, int ntasks,
               unsigned *err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    if ((smem_addr(sm) & 1023u) != 0) {  // the swizzled boxes need 1024-byte alignment
        if (threadIdx.x == 0) set_error(err, 0x4FF);
        return;
    }
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + kPrepStages * kPrepStage);
    uint64_t *empty = full + kPrepStages;
    volatile int *s_abort = reinterpret_cast<volatile int *>(empty + kPrepStages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = p.nQ * p.tile_q, groups = per / kPrepRows;
    const int mine = ntasks > (int)blockIdx.x ? (ntasks - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrepStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp >= kPrepConsumers) {
        if (lane == 0) {
            // --------------------------------------------------- producers
            // producer j issues tasks j, j + 2, ... into stages of parity j
            const int j = warp - kPrepConsumers;
            int issued[kPrepStages / kPrepProducers];
#pragma unroll
            for (int s = 0; s < kPrepStages / kPrepProducers; ++s) issued[s] = 0;
            tma_prefetch_desc(&tdo);
            tma_prefetch_desc(&to);
            for (int k = j; k < mine; k += kPrepProducers) {
                const int st = k % kPrepStages;
                if (k >= kPrepStages &&
                    !mbar_wait(empty + st, ((k / kPrepStages) - 1) & 1, s_abort, err, kSitePrepProd))
                    break;
                int b, h, s0;
                prep_task(p, (int)blockIdx.x + k * (int)gridDim.x, groups, b, h, s0);
                const int row = (p.layout == L_TND ? seq_start(p, true, b) : 0) + s0;
                const int bc = p.layout == L_TND ? 0 : b;
                uint8_t *dst = sm + st * kPrepStage;
                mbar_expect_tx(full + st, kPrepStage);
                tma_load_4d(dst, &tdo, full + st, 0, row, h, bc);
                tma_load_4d(dst + kPrepBox, &tdo, full + st, 64, row, h, bc);
                tma_load_4d(dst + 2 * kPrepBox, &to, full + st, 0, row, h, bc);
                tma_load_4d(dst + 3 * kPrepBox, &to, full + st, 64, row, h, bc);
                issued[st / kPrepProducers]++;
            }
            if (*s_abort) {  // drain this producer's copies before the CTA exits (bounded)
                int never = 0;
                for (int s = 0; s < kPrepStages / kPrepProducers; ++s)
                    if (issued[s])
                        mbar_wait(full + s * kPrepProducers + j, (issued[s] - 1) & 1, &never, nullptr, 0,
                                  200000000ull);
            }
        }
        return;
    }
    // ------------------------------------------------------------ consumers
    for (int k = warp; k < mine; k += kPrepConsumers) {
        const int st = k % kPrepStages;
        if (!__all_sync(0xffffffffu, mbar_wait(full + st, (k / kPrepStages) & 1, s_abort, err, kSitePrepCons)))
            break;
        int b, h, s0;
        prep_task(p, (int)blockIdx.x + k * (int)gridDim.x, groups, b, h, s0);
        // rows `lane` and `lane + 32` of the task: the two 64-column halves of dO and O
        const uint8_t *base = sm + st * kPrepStage;
        const float acc0 = prep_row_dot<T>(base, (uint32_t)lane);
        const float acc1 = prep_row_dot<T>(base, (uint32_t)lane + 32u);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + st);  // the stage's rows are in registers
        const int len = p.layout == L_TND ? seq_len(p, true, b) : per;
        const long long slot0 = ((long long)b * p.Hq + h) * per + s0;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int s = s0 + r * 32 + lane;
            const bool ex = s < len;
            ndvec[slot0 + r * 32 + lane] = ex ? -(r ? acc1 : acc0) : 0.f;
            const float lv = ex ? lse[lse_off(p, b, h, s)] : -INFINITY;
            nlse2[slot0 + r * 32 + lane] = lv == -INFINITY ? -INFINITY : -lv * kLog2e;  // a row with no key: P = 0
        }
    }
}

// ------------------------------------------------------ dK/dV order
// The dK/dV units differ in work by their KV-owned list lengths (a popular
// tile is listed by many query tiles), and the CTAs of one launch start in
// grid order. The units of one (batch entry, key/value head) share that
// head's Q and dO in L2, so the heads keep their grid order; within each
// head the longest units start first, which leaves the last head's short
// units for the end of the launch, where they fill the SMs that finish
// early (longest processing time first). A unit's key is the summed list
// length of its GQA group's heads (0 for a chunk without valid keys); a
// counting sort over kOrderBins bins of decreasing key (keys past the last
// bin share it) writes each head's part of the permutation. The order
// within a bin is the order of the atomics, which changes no result: each
// unit writes only its own dK, dV.
constexpr int kOrderBins = 1024, kOrderThreads = 1024;

// One CTA per (b, key/value head): units [seg * units_x, + units_x).
__global__ void __launch_bounds__(kOrderThreads) k_dk_order(const Prob p, const int *__restrict__ kv_ptr, int cap,
                                                           int *__restrict__ order, int *__restrict__ keys) {
    __shared__ int hist[kOrderBins];
    __shared__ int warp_sum[kOrderThreads / 32];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int subs_kv = p.tile_kv >> 7, units_x = p.nKV * subs_kv, g = p.Hq / p.Hkv;
    const int seg = blockIdx.x, hk = seg % p.Hkv, b = seg / p.Hkv;
    const long long base = (long long)seg * units_x;
    const int cap_all = p.nQ * cap;
    hist[t] = 0;
    __syncthreads();
    for (int x = t; x < units_x; x += kOrderThreads) {
        const int j = x / subs_kv, ck = x % subs_kv;
        int key = 0;
        if (kv_valid(p, b, j) > ck * 128)
            for (int h = hk * g; h < hk * g + g; ++h) {
                const int *ptr = kv_ptr + ((long long)b * p.Hq + h) * (p.nKV + 1);
                const int pos = clampi(ptr[j], 0, cap_all);
                key += clampi(ptr[j + 1], pos, cap_all) - pos;
            }
        const int bin = kOrderBins - 1 - min(key, kOrderBins - 1);  // bin 0: the longest
        keys[base + x] = bin;
        atomicAdd(&hist[bin], 1);
    }
    __syncthreads();
    // exclusive scan of the histogram (one bin per thread)
    const int v = hist[t];
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    if (lane == 31) warp_sum[w] = inc;
    __syncthreads();
    if (w == 0) {
        int s = warp_sum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        warp_sum[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    hist[t] = inc - v + (w > 0 ? warp_sum[w - 1] : 0);
    __syncthreads();
    for (int x = t; x < units_x; x += kOrderThreads)
        order[base + atomicAdd(&hist[keys[base + x]], 1)] = (int)(base + x);
}
static_assert(kOrderBins == kOrderThreads, "the scan takes one bin per thread");

// ----------------------------------------------------------- MMA helpers
// Measured on GB300 (all SMs busy, M = 128, K = 16 per instruction): an
// MMA with N = 128 takes 64 cycles with A from shared memory or from TMEM;
// N = 64 takes 45-48, ~70% of the N = 128 rate per FLOP. The dQ pass uses
// N = 128 throughout; the dK/dV pass's 64-row items make its S^T and dP^T
// MMAs N = 64 (the price of two TMEM buffers for them).

// D = A B^T, A and B [128 x 128] K-major 128-byte-swizzled tiles (two
// 64-column boxes 16 KB apart); 8 MMAs of K = 16.
__device__ __forceinline__ void issue_ss(uint32_t d, uint32_t aA, uint32_t aB, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t o = (kk >> 2) * kBox + (kk & 3) * 32;
        mma_f16_ss_w(d, sdesc_sw128(aA + o, 16, 1024), sdesc_sw128(aB + o, 16, 1024), idesc, kk > 0);
    }
}
// D (+)= A B with A [128 x 128] in TMEM (packed 16-bit pairs, 8 columns per
// K = 16) and B [K = 128 rows x N = 128] stored row-major (N contiguous),
// read MN-major (D halves 16 KB apart, 8-row groups 1 KB apart). KS = the
// K = 16 steps taken: 8, or 4 for the first 64 rows of B only.
template <int KS = 8>
__device__ __forceinline__ void issue_ts(uint32_t d, uint32_t a_tmem, uint32_t aB, uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = 0; kk < KS; ++kk)
        mma_f16_ts_w(d, a_tmem + kk * 8, sdesc_sw128(aB + kk * 2048, kBox, 1024), idesc, (acc || kk > 0) ? 1u : 0u);
}

// ----------------------------------------------------------------- dK/dV
// One CTA per (b, kv-head hk, 128-key chunk of KV tile j). K and V of the
// chunk stay in shared memory. Work items are the 64-row pieces of every
// query tile that selected j, over the query heads of hk's group, in
// (head, ascending tile, piece) order. Per item m:
//   S^T = K Q_m^T, dP^T = V dO_m^T        (128 keys x 64 rows, TMEM buffer m%2)
//   P^T = exp(scale S^T - LSE_t), dS^T = P^T (dP^T - Dvec_t)
//                                         (packed 16-bit, written back over
//                                          the consumed S^T / dP^T columns)
//   dV += P^T dO_m, dK += dS^T Q_m         (A operands read from TMEM)
// Two TMEM buffers let S^T / dP^T of item m+1 run on the tensor core while
// the softmax warps work on item m; each MMA warp's order is S/dP(0),
// S/dP(1), dV/dK(0), S/dP(2), dV/dK(1), S/dP(3), ... (S/dP(m+2) reuses the
// buffer that dV/dK(m), issued just before it, reads). One warp issues
// S^T and dV, another dP^T and dK.
// Eight softmax warps: warp w owns TMEM lanes 32*(w%4).. and the item's
// query columns 32*(w/4)..+31, and writes its packed results into the first
// 16 of those 32 columns, so no warp overwrites columns another still reads.
// TMEM columns: buffer x: S^T [128x, 128x+64) (P^T packed in [128x, +16)
// and [128x+32, +16)), dP^T [128x+64, 128x+128) (dS^T likewise);
// dV [256,384), dK [384,512).
constexpr int kDkStages = 4;
constexpr int kDkItem = 64;                // query rows per item
constexpr int kDkQTile = kDkItem * 256;    // one [64 x 128] 16-bit tile: two 8 KB boxes
constexpr int kDkQBox = kDkItem * 128;
constexpr int kDkOffK = 0, kDkOffV = kTile, kDkOffQ = 2 * kTile, kDkOffO = kDkOffQ + kDkStages * kDkQTile;
constexpr int kDkOffLd = kDkOffO + kDkStages * kDkQTile;  // per stage: nlse2[64], ndvec[64]
constexpr int kDkOffCtl = kDkOffLd + kDkStages * 512;
constexpr size_t kDkSmem = kDkOffCtl + 256;

// S^T = K Q_m^T (or dP^T = V dO_m^T): A = the 128-key tile, B = the 64-row
// tile, both K-major 128-byte-swizzled; N = 64.
__device__ __forceinline__ void issue_ss_n64(uint32_t d, uint32_t aA, uint32_t aB, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t o = (kk & 3) * 32;
        mma_f16_ss_w(d, sdesc_sw128(aA + (kk >> 2) * kBox + o, 16, 1024),
                     sdesc_sw128(aB + (kk >> 2) * kDkQBox + o, 16, 1024), idesc, kk > 0);
    }
}
// dV += P^T dO_m (or dK += dS^T Q_m): A in TMEM, K = 64 query rows packed in
// two 16-column pieces 32 columns apart (8 columns per K = 16 step); B = the
// 64-row tile read MN-major (D halves 8 KB apart, 8-row groups 1 KB apart).
__device__ __forceinline__ void issue_ts_k64(uint32_t d, uint32_t a_tmem, uint32_t aB, uint32_t idesc, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_f16_ts_w(d, a_tmem + (kk >> 1) * 32 + (kk & 1) * 8, sdesc_sw128(aB + kk * 2048, kDkQBox, 1024), idesc,
                     (acc || kk > 0) ? 1u : 0u);
}

struct WorkIter {
    int h, pos, end, sub, i, nsub;
};

// The KV-owned list of tile j for query head h: entries [pos, end) of
// kv_qidx. Offsets are clamped into [0, nQ * cap] with end >= pos and
// entries into [0, nQ), so a corrupt index (invalid input, reported by
// vsa_check_inputs) cannot move a read or a load outside its buffer.
__device__ __forceinline__ void kv_list(const Prob &p, const BwdArgs &a, int b, int h, int j, int &pos,
                                        int &end) {
    const int *ptr = a.kv_ptr + ((long long)b * p.Hq + h) * (p.nKV + 1);
    const int cap_all = p.nQ * a.cap;
    pos = clampi(ptr[j], 0, cap_all);
    end = clampi(ptr[j + 1], pos, cap_all);
}
__device__ __forceinline__ int kv_entry(const Prob &p, const BwdArgs &a, int b, int h, int pos) {
    return clampi(a.kv_qidx[((long long)b * p.Hq + h) * p.nQ * a.cap + pos], 0, p.nQ - 1);
}

__device__ __forceinline__ bool work_next_list(const Prob &p, const BwdArgs &a, int b, int h_end, int j,
                                               WorkIter &w) {
    while (w.pos >= w.end) {
        if (++w.h >= h_end) return false;
        kv_list(p, a, b, w.h, j, w.pos, w.end);
    }
    w.i = kv_entry(p, a, b, w.h, w.pos);
    w.nsub = (q_rows(p, b, w.i) + kDkItem - 1) / kDkItem;
    w.sub = 0;
    return true;
}
__device__ __forceinline__ bool work_first(const Prob &p, const BwdArgs &a, int b, int h0, int h_end, int j,
                                           WorkIter &w) {
    w.h = h0;
    kv_list(p, a, b, h0, j, w.pos, w.end);
    return work_next_list(p, a, b, h_end, j, w);
}
__device__ __forceinline__ bool work_advance(const Prob &p, const BwdArgs &a, int b, int h_end, int j,
                                             WorkIter &w) {
    if (++w.sub < w.nsub) return true;
    ++w.pos;
    return work_next_list(p, a, b, h_end, j, w);
}

template <typename T>
__global__ void __launch_bounds__(kDkThreads, 1)
    k_dkdv(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
           const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
           const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv, const Prob p,
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
    uint64_t *b_pd = b_sf + 2, *b_acc = b_pd + 2, *b_fin = b_acc + 1;  // b_fin: one per MMA warp
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(b_fin + 2);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nwork = reinterpret_cast<int *>(s_tmem + 2);
    // per stage: the item's query-block bits and its 64-row piece index
    int *s_item = reinterpret_cast<int *>(sm + kDkOffCtl + 160);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int subs_kv = p.tile_kv >> 7;
    // this CTA's unit: the launch order is longest work first (an order
    // entry out of range is invalid input and is clamped into the grid)
    const int units_x = p.nKV * subs_kv;
    const int u = a.dk_order ? clampi(a.dk_order[blockIdx.x], 0, (int)gridDim.x - 1) : (int)blockIdx.x;
    const int x = u % units_x, j = x / subs_kv, ck = x % subs_kv;
    const int hk = (u / units_x) % p.Hkv, b = u / (units_x * p.Hkv), g = p.Hq / p.Hkv;
    const int h0 = hk * g, h_end = h0 + g;
    const int kvalid_tile = kv_valid(p, b, j);
    int kvalid = kvalid_tile - ck * 128;
    kvalid = kvalid < 0 ? 0 : (kvalid > 128 ? 128 : kvalid);
    const int key0 = j * p.tile_kv + ck * 128;  // within the batch entry
    if (p.layout == L_TND && kvalid == 0) return;  // keys outside the sequence do not exist
    const int kvb = (p.layout == L_TND ? seq_start(p, false, b) : 0), qb = (p.layout == L_TND ? seq_start(p, true, b) : 0);
    const int bc = (p.layout == L_TND ? 0 : b);

    if (threadIdx.x == 0) {
        mbar_init(b_kv, 1);
        for (int s = 0; s < kDkStages; ++s) {
            mbar_init(b_qf + s, 1);
            mbar_init(b_qe + s, 2);  // both MMA warps
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_sf + x, 2);  // both MMA warps
            mbar_init(b_pd + x, 256);
            mbar_init(b_fin + x, 1);
        }
        mbar_init(b_acc, 2);
        *s_abort = 0;
        // count the work items (a chunk with no valid key does no work)
        int n = 0;
        if (kvalid > 0)
            for (int h = h0; h < h_end; ++h) {
                int pos, end;
                kv_list(p, a, b, h, j, pos, end);
                if (p.layout != L_TND) {  // every query tile has tile_q rows
                    n += (end - pos) * (p.tile_q / kDkItem);
                    continue;
                }
                for (int q = pos; q < end; ++q) n += (q_rows(p, b, kv_entry(p, a, b, h, q)) + kDkItem - 1) / kDkItem;
            }
        *s_nwork = n;
        fence_mbar_init();
    }
    // the producer's first work item is looked up while thread 0 counts
    WorkIter w{};
    bool more = false;
    if (warp == kProdWarp && lane == 0 && kvalid > 0) more = work_first(p, a, b, h0, h_end, j, w);
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
        for (int m = 0; more && m < M; ++m) {
            const int st = m % kDkStages;
            if (m >= kDkStages && !mbar_wait(b_qe + st, ((m / kDkStages) - 1) & 1, s_abort, a.err, kSiteDkProd))
                break;
            const int row = qb + w.i * p.tile_q + w.sub * kDkItem;
            const long long slot =
                ((long long)b * p.Hq + w.h) * p.nQ * p.tile_q + w.i * p.tile_q + w.sub * kDkItem;
            if (a.kv_qsub) {  // read by the softmax after this stage's barrier completes
                s_item[2 * st] = a.kv_qsub[((long long)b * p.Hq + w.h) * p.nQ * a.cap + w.pos];
                s_item[2 * st + 1] = w.sub;
            }
            mbar_expect_tx(b_qf + st, 2 * kDkQTile + 512);
            tma_load_4d(sQ + st * kDkQTile, &tq, b_qf + st, 0, row, w.h, bc);
            tma_load_4d(sQ + st * kDkQTile + kDkQBox, &tq, b_qf + st, 64, row, w.h, bc);
            tma_load_4d(sO + st * kDkQTile, &tdo, b_qf + st, 0, row, w.h, bc);
            tma_load_4d(sO + st * kDkQTile + kDkQBox, &tdo, b_qf + st, 64, row, w.h, bc);
            bulk_load(sLd + st * 512, a.nlse2 + slot, 256, b_qf + st);
            bulk_load(sLd + st * 512 + 256, a.ndvec + slot, 256, b_qf + st);
            issued[st]++;
            more = work_advance(p, a, b, h_end, j, w);
        }
    } else if ((warp == kMmaWarp || warp == kDkMma2Warp) && M > 0) {
        // -------------------------------- MMA issuers (two whole warps, one lane each)
        // Warp 0 of the pair: S^T = K Q^T and dV += P^T dO; warp 1: dP^T =
        // V dO^T and dK += dS^T Q. Each warp's accumulation reads only the
        // columns its own score MMA wrote, and S/dP(m+2) overwrites what
        // dV/dK(m) of the same warp reads, issued just before; so the two
        // warps share no TMEM hazard and their waits overlap each other's MMAs.
        const int mw = warp == kMmaWarp ? 0 : 1;
        const uint32_t idS = idesc_f16(bf16, 128, 64, false, false);
        const uint32_t idA = idesc_f16(bf16, 128, 128, false, true);
        const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aQ = smem_addr(sQ), aO = smem_addr(sO);
        const uint32_t aX = mw ? aV : aK;     // scores: A operand
        const uint32_t aS = mw ? aO : aQ;     // scores: B operand (per stage)
        const uint32_t aG = mw ? aQ : aO;     // accumulation: B operand (per stage)
        const uint32_t tAcc = tbase + 256 + mw * 128, off = mw * 64;
        bool ok = mbar_wait_warp(b_kv, 0, s_abort, a.err, kSiteDkMma);
        // scores of items 0 and 1
        for (int m = 0; ok && m < 2 && m < M; ++m) {
            if (!(ok = mbar_wait_warp(b_qf + m, 0, s_abort, a.err, kSiteDkMma))) break;
            tc_fence_after();
            issue_ss_n64(tbase + m * 128 + off, aX, aS + m * kDkQTile, idS);
            mma_commit_w(b_sf + m);
            mma_started = 1;
        }
        for (int m = 0; ok && m < M; ++m) {
            const int x = m & 1, st = m % kDkStages;
            const uint32_t tx = tbase + x * 128 + off;
            if (!(ok = mbar_wait_warp(b_pd + x, (m >> 1) & 1, s_abort, a.err, kSiteDkMma))) break;
            tc_fence_after();
            issue_ts_k64(tAcc, tx, aG + st * kDkQTile, idA, m > 0);  // dV += P^T dO | dK += dS^T Q
            mma_commit_w(b_qe + st);
            const int n = m + 2;
            if (n < M) {
                const int sn = n % kDkStages;
                if (!(ok = mbar_wait_warp(b_qf + sn, (n / kDkStages) & 1, s_abort, a.err, kSiteDkMma))) break;
                tc_fence_after();
                issue_ss_n64(tx, aX, aS + sn * kDkQTile, idS);
                mma_commit_w(b_sf + x);
            }
        }
        if (ok) mma_commit_w(b_acc);
    } else if (warp < 8) {
        // ------------------------------------------- softmax + epilogue
        const int lg = warp & 3, ch = warp >> 2;  // lane quarter, query-column half
        const int u = lg * 32 + lane;             // key row within the chunk
        const uint32_t tl = tbase + ((uint32_t)(lg * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        const bool key_ok = u < kvalid;
        bool ok = true;
        for (int m = 0; m < M; ++m) {
            const int x = m & 1, st = m % kDkStages;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(b_sf + x, (m >> 1) & 1, s_abort, a.err, kSiteDkSoft) &&
                                mbar_wait(b_qf + st, (m / kDkStages) & 1, s_abort, a.err, kSiteDkSoft));
            if (!ok) break;
            tc_fence_after();
            // this warp's 32 query columns of S^T and dP^T
            const uint32_t cs = x * 128 + ch * 32;
            uint32_t sr[32], dr[32];
            tmem_ld32(tl + cs, sr);
            tmem_ld32(tl + cs + 64, dr);
            tmem_wait_ld();
            if (!key_ok) {  // keys past the chunk's valid count: P^T = 0
#pragma unroll
                for (int e = 0; e < 32; ++e) sr[e] = __float_as_uint(-INFINITY);
            }
            // query blocks that did not select this tile: P^T = 0 in their
            // columns (block_q is a multiple of 32, so this warp's 32 columns
            // lie in one block)
            if (a.kv_qsub && !((s_item[2 * st] >> ((s_item[2 * st + 1] * kDkItem + ch * 32) / a.block_q)) & 1)) {
#pragma unroll
                for (int e = 0; e < 32; ++e) sr[e] = __float_as_uint(-INFINITY);
            }
            // P^T = 2^(scale log2e S^T + nlse2_t), dS^T = P^T (dP^T + ndvec_t), on pairs
            const ulonglong2 *nl = reinterpret_cast<const ulonglong2 *>(sLd + st * 512) + ch * 8;
            const ulonglong2 *nd = reinterpret_cast<const ulonglong2 *>(sLd + st * 512 + 256) + ch * 8;
            const uint64_t sc2 = f32x2(sl2, sl2);
            uint32_t pw[16], dw[16];
#pragma unroll
            for (int t4 = 0; t4 < 8; ++t4) {
                const ulonglong2 l4 = nl[t4], d4 = nd[t4];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int e = t4 * 4 + hh * 2;
                    const float2 xx = f32x2_split(
                        ffma_x2(f32x2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2, hh ? l4.y : l4.x));
                    const float p0 = ex2(xx.x), p1 = ex2(xx.y);
                    const float2 dd = f32x2_split(fmul_x2(
                        f32x2(p0, p1), fadd_x2(f32x2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                               hh ? d4.y : d4.x)));
                    pw[t4 * 2 + hh] = pack2<T>(p0, p1);
                    dw[t4 * 2 + hh] = pack2<T>(dd.x, dd.y);
                }
            }
            // into this warp's own, already read columns
            tmem_st16(tl + cs, pw);
            tmem_st16(tl + cs + 64, dw);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_pd + x);
        }
        if (ok && M > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_acc, 0, s_abort, a.err, kSiteDkSoft));
            if (ok) tc_fence_after();
        }
        const bool have = ok && M > 0;
        const bool row_ok = (p.layout == L_TND) ? key_ok : true;
        const long long ro = tok_off(p, false, b, key0 + u, hk);
        T *dst = reinterpret_cast<T *>(ch ? a.dk : a.dv) + ro;   // half 0 writes dV, half 1 dK
        const float inv = kvalid_tile > 0 ? 1.f / (float)kvalid_tile : 0.f;
        const float *cbase = ch ? a.dpk : a.dpv;
        const float *cadd = cbase ? cbase + (((long long)b * p.Hkv + hk) * p.nKV + j) * 128 : nullptr;
        const float mul = ch ? p.scale : 1.f;
        // Padded layouts: the chunk's 128 rows of dV and dK are staged in the
        // Q stages (free once every accumulation MMA is done) in the TMA box
        // layout and stored by four box copies, instead of 16-byte stores
        // that each touch 32 rows. A varlen chunk may end inside its tile
        // (its last rows belong to the next sequence): per-thread stores.
        const bool staged = p.layout != L_TND;
        uint8_t *stage = sQ + ch * 2 * kBox;  // [2 boxes of 64 dims][128 rows x 128 B]
#pragma unroll 1
        for (int q8 = 0; q8 < 2; ++q8) {
            uint32_t o2[2][32];  // two quarters per TMEM round trip
            if (have) {
                tmem_ld32(tl + 256 + ch * 128 + q8 * 64, o2[0]);
                tmem_ld32(tl + 256 + ch * 128 + q8 * 64 + 32, o2[1]);
                tmem_wait_ld_regs(o2[0]);
                tmem_wait_ld_regs(o2[1]);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o2[0][e] = o2[1][e] = 0u;
            }
            if (!row_ok) continue;
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                const int q4 = q8 * 2 + hq;
                const uint32_t(&o)[32] = o2[hq];
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
                if (staged) {
                    // dims q4*32 .. +31: box q4 / 2, 16-byte chunks 4 (q4 % 2) .. +3 of row u, 128-byte swizzle
                    uint8_t *rowp = stage + (q4 >> 1) * kBox + u * 128;
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        *reinterpret_cast<uint4 *>(rowp + ((((q4 & 1) * 4 + t) ^ (u & 7)) << 4)) =
                            make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
                } else {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + q4 * 32);
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        d4[t] = make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
                }
            }
        }
        if (staged) {
            fence_proxy_async_smem();
            named_sync(1, 256);  // the 8 epilogue warps have staged their rows
            if (warp == 0 && lane == 0 && !*s_abort) {
                for (int t = 0; t < 2; ++t) {
                    tma_store_4d(t ? &tdk : &tdv, sQ + t * 2 * kBox, 0, key0, hk, bc);
                    tma_store_4d(t ? &tdk : &tdv, sQ + t * 2 * kBox + kBox, 64, key0, hk, bc);
                }
                tma_store_commit();
                tma_store_wait_read();  // the stage is read before this CTA's shared memory goes
            }
        }
    }

    if (*s_abort) {
        int never = 0;
        if (warp == kProdWarp && lane == 0) {
            if (issued_kv) mbar_wait(b_kv, 0, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < kDkStages; ++s)
                if (issued[s]) mbar_wait(b_qf + s, (issued[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
        }
    }
    if ((warp == kMmaWarp || warp == kDkMma2Warp) && mma_started && __any_sync(0xffffffffu, *s_abort != 0)) {
        // the MMAs this warp issued finish before TMEM is released
        int never = 0;
        const int mw = warp == kMmaWarp ? 0 : 1;
        mma_commit_w(b_fin + mw);
        __all_sync(0xffffffffu, mbar_wait(b_fin + mw, 0, &never, nullptr, 0, 200000000ull));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// -------------------------------------------------------------------- dQ
// One CTA per (b, h, 128-row chunk of query tile i), looping over the
// selected KV tiles' 128-key chunks:
//   S = Q K^T, dP = dO V^T (TMEM), P = exp(scale S - LSE),
//   dS = P (dP - Dvec) -> TMEM (packed, two buffers), dQ += dS K (TMEM).
// The eight softmax warps (lane quarter x key-column half) read S and dP
// into registers and release them at once, so S/dP of the next chunk run
// on the tensor core while this chunk's dS is computed; dQ += dS K reads
// dS from TMEM. Three warps issue MMAs: S(c), dP(c) and dQ(c) (once dS(c)
// is written) each from their own, so the synchronisation of one warp
// overlaps the others' MMAs. K chunks stay until dQ += dS K has read them,
// one chunk after S, so K has three stages; V, free right after dP, has
// two. The chunk sequence (selected tiles in ascending order, each cut into
// 128-key chunks with valid keys) is walked from a per-warp window of the
// index, not stored.
// TMEM columns: S [0,128), dP [128,256), dQ [256,384), dS buffers
// [384,448) and [448,512).
constexpr int kDqKStages = 3, kDqVStages = 2;
constexpr int kDqOffQ = 0, kDqOffO = kTile, kDqOffK = 2 * kTile, kDqOffV = (2 + kDqKStages) * kTile;
constexpr int kDqOffCtl = kDqOffV + kDqVStages * kTile;
constexpr int kDqOffHalf = kDqOffCtl + 256;  // one bit per chunk: at most 64 valid keys
constexpr size_t kDqSmem = kDqOffHalf + kMaxChunks / 8;
static_assert(kDqSmem <= 232448, "dQ shared memory exceeds the 227 KB a CTA may use");

template <typename T>
__global__ void __launch_bounds__(kDqThreads, 1)
    k_dq(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
         const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
         const __grid_constant__ CUtensorMap tdq, const Prob p, const BwdArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    if ((smem_addr(sm) & 1023u) != 0) {
        if (threadIdx.x == 0) set_error(a.err, 0x3FF);
        return;
    }
    uint8_t *sQ = sm + kDqOffQ, *sO = sm + kDqOffO, *sK = sm + kDqOffK, *sV = sm + kDqOffV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kDqOffCtl);
    uint64_t *b_q = bars + 0, *b_kf = bars + 1, *b_ke = bars + 4, *b_vf = bars + 7, *b_ve = bars + 9;
    // b_sf / b_sfree: [0] for S, [1] for dP (each computed, then read, on its own)
    uint64_t *b_sf = bars + 11, *b_sfree = bars + 13, *b_dsf = bars + 15, *b_dq = bars + 17;
    uint64_t *b_fin = bars + 19;  // one per MMA warp
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 22);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    int *s_nchunk = reinterpret_cast<int *>(s_tmem + 2);
    unsigned *s_half = reinterpret_cast<unsigned *>(sm + kDqOffHalf);  // [kMaxChunks / 32]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int subs = p.tile_q >> 7;
    const int i = blockIdx.x / subs, half = blockIdx.x % subs;
    const int h = blockIdx.y, b = blockIdx.z, hk = h / (p.Hq / p.Hkv);
    const int row0 = i * p.tile_q + half * 128;
    int nrows = 128;
    if (p.layout == L_TND) {
        nrows = seq_len(p, true, b) - row0;
        if (nrows <= 0) return;
        nrows = nrows > 128 ? 128 : nrows;
    }
    const int qrc = (p.layout == L_TND ? seq_start(p, true, b) : 0) + row0;
    const int kvb = (p.layout == L_TND ? seq_start(p, false, b) : 0);
    const int bc = (p.layout == L_TND ? 0 : b);
    const long long qrow = ((long long)b * p.Hq + h) * p.nQ + i;

    if (threadIdx.x == 0) {
        mbar_init(b_q, 1);
        for (int s = 0; s < kDqKStages; ++s) {
            mbar_init(b_kf + s, 1);
            mbar_init(b_ke + s, 1);
        }
        for (int s = 0; s < kDqVStages; ++s) {
            mbar_init(b_vf + s, 1);
            mbar_init(b_ve + s, 1);
        }
        for (int s = 0; s < 2; ++s) mbar_init(b_dq + s, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(b_sf + s, 1);
            mbar_init(b_sfree + s, 256);
        }
        for (int s = 0; s < 2; ++s) mbar_init(b_dsf + s, 256);
        for (int s = 0; s < 3; ++s) mbar_init(b_fin + s, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    // The producer reads the selection before the CTA-wide sync: the chunk
    // count and bits every role needs, and the first window of its own
    // walk, so that Q, dO and the first K/V chunk are requested right after.
    ChunkWin pcw{};
    if (warp == kProdWarp) {
        // number of 128-key chunks with valid keys (counts clamped to
        // idx_cap, tile ids outside [0, nKV) skipped, as in win_load)
        // and, per chunk, whether it holds at most 64 valid keys (then its
        // MMAs run over the first 64 keys only)
        const int *idx = a.q_idx + qrow * a.cap;
        // the row's first 32 entries are read without waiting for their
        // count (a row holds idx_cap entries), so the two reads overlap
        const int jfirst = lane < a.cap ? idx[lane] : -1;
        const int cnt = clampi(a.q_cnt[qrow], 0, a.cap);
        const int per = p.tile_kv >> 7;
        for (int x = lane; x < kMaxChunks / 32; x += 32) s_half[x] = 0u;
        __syncwarp();
        int total = 0;  // chunks of the entries before this group of 32
        for (int n0 = 0; n0 < cnt; n0 += 32) {
            const int n = n0 + lane, j = n < cnt ? (n0 == 0 ? jfirst : idx[n]) : -1;
            const int kvv = (j >= 0 && j < p.nKV) ? kv_valid(p, b, j) : 0;
            const int nch = min(per, (kvv + 127) >> 7);
            int inc = nch;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += y;
            }
            for (int k = 0, ci = total + inc - nch; k < nch; ++k, ++ci)
                if (ci < kMaxChunks && kvv - k * 128 <= 64) atomicOr(&s_half[ci >> 5], 1u << (ci & 31));
            total += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) *s_nchunk = min(total, kMaxChunks);
        pcw = win_begin(p, b, idx, nullptr, cnt, lane);
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
    int issued_q = 0, issued_k[kDqKStages] = {0, 0, 0}, issued_v[kDqVStages] = {0, 0}, mma_started = 0;

    if (warp == kProdWarp && N > 0) {
        // ------------------------------------ TMA producer (whole warp, lane 0 issues)
        ChunkWin &cw = pcw;
        if (lane == 0) {
            mbar_expect_tx(b_q, 2 * kTile);
            tma_load_4d(sQ, &tq, b_q, 0, qrc, h, bc);
            tma_load_4d(sQ + kBox, &tq, b_q, 64, qrc, h, bc);
            tma_load_4d(sO, &tdo, b_q, 0, qrc, h, bc);
            tma_load_4d(sO + kBox, &tdo, b_q, 64, qrc, h, bc);
        }
        issued_q = 1;
        for (int c = 0; c < N; ++c) {
            int crow = 0, cval = 0, cbits = -1;
            if (!win_chunk(p, b, cw, c, lane, crow, cval, cbits)) break;
            const int sk = c % kDqKStages, sv = c % kDqVStages;
            const int kr = kvb + crow;
            // V first: its stage frees when dP(c-2) completes, which precedes
            // dQ(c-3), the MMA that frees K's stage
            if (c >= kDqVStages &&
                !mbar_wait_warp(b_ve + sv, ((c / kDqVStages) - 1) & 1, s_abort, a.err, kSiteDqProd))
                break;
            if (lane == 0) {
                mbar_expect_tx(b_vf + sv, kTile);
                tma_load_4d(sV + sv * kTile, &tv, b_vf + sv, 0, kr, hk, bc);
                tma_load_4d(sV + sv * kTile + kBox, &tv, b_vf + sv, 64, kr, hk, bc);
            }
            issued_v[sv]++;
            if (c >= kDqKStages &&
                !mbar_wait_warp(b_ke + sk, ((c / kDqKStages) - 1) & 1, s_abort, a.err, kSiteDqProd))
                break;
            if (lane == 0) {
                mbar_expect_tx(b_kf + sk, kTile);
                tma_load_4d(sK + sk * kTile, &tk, b_kf + sk, 0, kr, hk, bc);
                tma_load_4d(sK + sk * kTile + kBox, &tk, b_kf + sk, 64, kr, hk, bc);
            }
            issued_k[sk]++;
        }
    } else if ((warp == kMmaWarp || warp == kDqPMmaWarp) && N > 0) {
        // ------------------------- S issuer (warp 9) and dP issuer (warp 11)
        // S(c) needs only S(c-1) read out, dP(c) only dP(c-1); with a warp
        // each, the read of one overlaps the other's MMAs.
        const bool isP = warp == kDqPMmaWarp;
        const uint32_t idS = idesc_f16(bf16, 128, 128, false, false);
        const uint32_t idS64 = idesc_f16(bf16, 128, 64, false, false);  // chunks of at most 64 valid keys
        const uint32_t aA = smem_addr(isP ? sO : sQ), aB = smem_addr(isP ? sV : sK);
        const uint32_t tD = tbase + (isP ? 128 : 0);
        const int nst = isP ? kDqVStages : kDqKStages;
        uint64_t *b_full = isP ? b_vf : b_kf;
        bool ok = mbar_wait_warp(b_q, 0, s_abort, a.err, kSiteDqMma);
        unsigned hw = 0u;  // the chunk bits of c's word, read once per 32 chunks ahead of the waits
        for (int c = 0; ok && c < N; ++c) {
            const int sx = c % nst;
            if ((c & 31) == 0) hw = s_half[c >> 5];
            const bool hc = (hw >> (c & 31)) & 1u;
            if (!(ok = mbar_wait_warp(b_full + sx, (c / nst) & 1, s_abort, a.err, kSiteDqMma))) break;
            if (c > 0 && !(ok = mbar_wait_warp(b_sfree + isP, (c - 1) & 1, s_abort, a.err, kSiteDqMma))) break;
            tc_fence_after();
            // S = Q K^T | dP = dO V^T, over the chunk's first 64 keys when no
            // others are valid (a branch, so each form keeps its descriptor constant)
            if (hc)
                issue_ss(tD, aA, aB + sx * kTile, idS64);
            else
                issue_ss(tD, aA, aB + sx * kTile, idS);
            mma_commit_w(b_sf + isP);
            if (isP) mma_commit_w(b_ve + sx);  // V_c free once dP(c) is done
            mma_started = 1;
        }
    } else if (warp == kDqMmaWarp && N > 0) {
        // --------------------------------------------- dQ issuer (whole warp)
        // Its MMAs touch no TMEM columns or stages the S / dP issuer writes,
        // so the two warps issue independently; the waits of one overlap
        // the other's MMAs.
        const uint32_t idQ = idesc_f16(bf16, 128, 128, false, true);
        const uint32_t aK = smem_addr(sK);
        const uint32_t tQ = tbase + 256, tX = tbase + 384;
        bool ok = true;
        unsigned hw = 0u;  // as for the S / dP issuers
        for (int c = 0; ok && c < N; ++c) {
            const int sk = c % kDqKStages;
            if ((c & 31) == 0) hw = s_half[c >> 5];
            const bool hc = (hw >> (c & 31)) & 1u;
            if (!(ok = mbar_wait_warp(b_dsf + (c & 1), (c >> 1) & 1, s_abort, a.err, kSiteDqMma))) break;
            tc_fence_after();
            if (hc)  // dQ += dS K over the first 64 keys (the rest are not valid)
                issue_ts<4>(tQ, tX + (c & 1) * 64, aK + sk * kTile, idQ, c > 0);
            else
                issue_ts(tQ, tX + (c & 1) * 64, aK + sk * kTile, idQ, c > 0);  // dQ += dS K
            mma_commit_w(b_dq + (c & 1));
            mma_commit_w(b_ke + sk);
            mma_started = 1;
        }
    } else if (warp < 8) {
        const int lg = warp & 3, ch = warp >> 2;  // lane quarter, key-column half
        const int r = lg * 32 + lane;
        const uint32_t tl = tbase + ((uint32_t)(lg * 32) << 16);
        const float sl2 = p.scale * kLog2e;
        const bool row_ok = r < nrows;
        const long long slot = ((long long)b * p.Hq + h) * p.nQ * p.tile_q + row0 + r;
        const float nl2 = N > 0 ? a.nlse2[slot] : -INFINITY;
        const float ndv = N > 0 ? a.ndvec[slot] : 0.f;
        bool ok = true;
        ChunkWin cw = win_begin(p, b, a.q_idx + qrow * a.cap, a.q_sub ? a.q_sub + qrow * a.cap : nullptr,
                                clampi(a.q_cnt[qrow], 0, a.cap), lane);
        // The chunk loop is instantiated twice: with the half-chunk skip
        // below, for query tiles that selected a chunk of at most 64 valid
        // keys, and without it, so that the other tiles run a loop whose
        // code the skip does not change.
        auto chunks = [&](auto with_half) {
            for (int c = 0; c < N; ++c) {
                int crow = 0, cval = 0, cbits = -1;
                win_chunk(p, b, cw, c, lane, crow, cval, cbits);
                int valid = cval - ch * 64;
                // query blocks: a row whose block did not select this tile sees no key of it
                if (a.q_sub && !((cbits >> ((half * 128 + r) / a.block_q)) & 1)) valid = 0;
                uint32_t sr[64], dr[64];
                ok = __all_sync(0xffffffffu, mbar_wait(b_sf, c & 1, s_abort, a.err, kSiteDqSoft));
                if (!ok) break;
                tc_fence_after();
                tmem_ld32(tl + ch * 64, *reinterpret_cast<uint32_t(*)[32]>(sr));
                tmem_ld32(tl + ch * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(b_sfree);  // S of this chunk is in registers
                ok = __all_sync(0xffffffffu, mbar_wait(b_sf + 1, c & 1, s_abort, a.err, kSiteDqSoft));
                if (!ok) break;
                tc_fence_after();
                tmem_ld32(tl + 128 + ch * 64, *reinterpret_cast<uint32_t(*)[32]>(dr));
                tmem_ld32(tl + 128 + ch * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(b_sfree + 1);  // and dP
                // A chunk of at most 64 valid keys runs N = 64 MMAs (no S, dP for
                // keys 64..127, which the loads above read as stale columns) and
                // a dQ MMA over the first 64 keys only: the warps of the key half
                // 64..127 write no dS. They still take every barrier in step, so
                // no arrival of theirs can count towards another chunk's phase.
                if constexpr (decltype(with_half)::value) {
                    if (ch == 1 && cval <= 64) {
                        mbar_arrive(b_dsf + (c & 1));
                        continue;
                    }
                }
                if (valid < 64) {  // keys past the valid count: P = 0
#pragma unroll
                    for (int kk = 0; kk < 64; ++kk)
                        if (kk >= valid) sr[kk] = __float_as_uint(-INFINITY);
                }
                // P = 2^(S scale log2e - LSE log2e), dS = P (dP - Dvec), on pairs
                const uint64_t sc2 = f32x2(sl2, sl2), nl2x = f32x2(nl2, nl2), nd2 = f32x2(ndv, ndv);
                uint32_t dw[32];
#pragma unroll
                for (int t2 = 0; t2 < 32; ++t2) {
                    const float2 x = f32x2_split(
                        ffma_x2(f32x2(__uint_as_float(sr[2 * t2]), __uint_as_float(sr[2 * t2 + 1])), sc2, nl2x));
                    const uint64_t pp = f32x2(ex2(x.x), ex2(x.y));
                    const uint64_t dd = fmul_x2(pp, fadd_x2(f32x2(__uint_as_float(dr[2 * t2]), __uint_as_float(dr[2 * t2 + 1])), nd2));
                    const float2 d2 = f32x2_split(dd);
                    dw[t2] = pack2<T>(d2.x, d2.y);
                }
                if (c >= 2) {  // dS buffer c&1 was read by dQ(c-2)
                    ok = __all_sync(0xffffffffu, mbar_wait(b_dq + (c & 1), ((c >> 1) - 1) & 1, s_abort, a.err,
                                                           kSiteDqSoft));
                    if (!ok) break;
                    tc_fence_after();
                }
                tmem_st32(tl + 384 + (c & 1) * 64 + ch * 32, dw);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(b_dsf + (c & 1));
            }
        };
        unsigned any_half = 0u;
        for (int x = 0; x < (N + 31) / 32; ++x) any_half |= s_half[x];
        if (any_half)
            chunks(std::true_type{});
        else
            chunks(std::false_type{});
        if (ok && N > 0) {
            const int cp = N - 1;
            ok = __all_sync(0xffffffffu, mbar_wait(b_dq + (cp & 1), (cp >> 1) & 1, s_abort, a.err, kSiteDqSoft));
            if (ok) tc_fence_after();
        }
        const bool have = ok && N > 0;
        const long long ro = tok_off(p, true, b, row0 + r, h) + ch * 64;
        T *dq = reinterpret_cast<T *>(a.dq) + ro;
        const int qv = a.dpq ? q_valid(p, b, i) : 0;
        const bool add_c = a.dpq && (half * 128 + r) < qv;
        const float *cq = a.dpq ? a.dpq + qrow * 128 + ch * 64 : nullptr;
        const float inv = qv > 0 ? 1.f / (float)qv : 0.f;
        // Padded layouts: the chunk's 128 rows of dQ are staged in the Q tile
        // (free once the last S MMA is done) in the TMA box layout and stored
        // by two box copies; varlen rows past the sequence must not be
        // written, so there each thread stores its own row.
        const bool staged = p.layout != L_TND;
#pragma unroll 1
        for (int q2 = 0; q2 < 2; ++q2) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tl + 256 + ch * 64 + q2 * 32, o);
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
                    v0 += cq[q2 * 32 + 2 * e2] * inv;
                    v1 += cq[q2 * 32 + 2 * e2 + 1] * inv;
                }
                wv[e2] = pack2<T>(v0, v1);
            }
            if (staged) {
                // columns 64 ch + 32 q2 .. +31: box ch, 16-byte chunks 4 q2 .. +3 of row r, 128-byte swizzle
                uint8_t *rowp = sQ + ch * kBox + r * 128;
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    *reinterpret_cast<uint4 *>(rowp + (((q2 * 4 + t) ^ (r & 7)) << 4)) =
                        make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
            } else {
                uint4 *d4 = reinterpret_cast<uint4 *>(dq + q2 * 32);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    d4[t] = make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
            }
        }
        if (staged) {
            fence_proxy_async_smem();
            named_sync(1, 256);  // the 8 epilogue warps have staged their rows
            if (warp == 0 && lane == 0 && !*s_abort) {
                tma_store_4d(&tdq, sQ, 0, qrc, h, bc);
                tma_store_4d(&tdq, sQ + kBox, 64, qrc, h, bc);
                tma_store_commit();
                tma_store_wait_read();  // the stage is read before this CTA's shared memory goes
            }
        }
    }

    if (*s_abort) {
        int never = 0;
        if (warp == kProdWarp && lane == 0) {
            if (issued_q) mbar_wait(b_q, 0, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < kDqKStages; ++s)
                if (issued_k[s]) mbar_wait(b_kf + s, (issued_k[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
            for (int s = 0; s < kDqVStages; ++s)
                if (issued_v[s]) mbar_wait(b_vf + s, (issued_v[s] - 1) & 1, &never, nullptr, 0, 200000000ull);
        }
    }
    if ((warp == kMmaWarp || warp == kDqMmaWarp || warp == kDqPMmaWarp) && mma_started &&
        __any_sync(0xffffffffu, *s_abort != 0)) {
        // the MMAs this warp issued finish before TMEM is released
        int never = 0;
        mma_commit_w(b_fin + (warp - kMmaWarp));
        __all_sync(0xffffffffu, mbar_wait(b_fin + (warp - kMmaWarp), 0, &never, nullptr, 0, 200000000ull));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

}  // namespace

namespace {

// dgate of the gated compression branch: out_t = O_t + gate_t (*) c_i for
// every slot t of query tile i, so dgate_t = dO_t (*) c_i (fp32 product,
// rounded once). A half-warp per (b, slot, head) row, 16 bytes per thread;
// in TND only rows inside a sequence exist.
template <typename T>
__global__ void __launch_bounds__(256) k_gate_grad(Prob p, const T *__restrict__ dO, const float *__restrict__ c,
                                                   T *__restrict__ dgate) {
    const int sub = threadIdx.x & 15;
    const long long slots = (long long)p.nQ * p.tile_q;
    const long long per_b = slots * p.Hq;
    const long long units = (long long)p.B * per_b;
    const long long step = ((long long)gridDim.x * blockDim.x) >> 4;
    for (long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 4; u < units; u += step) {
        const int b = (int)(u / per_b);
        const long long rem = u - (long long)b * per_b;
        const int s = (int)(rem / p.Hq), h = (int)(rem % p.Hq);
        if (p.layout == L_TND && s >= seq_len(p, true, b)) continue;
        const long long o = tok_off(p, true, b, s, h) + sub * 8;
        const float *cc = c + (((long long)b * p.Hq + h) * p.nQ + s / p.tile_q) * 128 + sub * 8;
        const uint4 g = *reinterpret_cast<const uint4 *>(dO + o);
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t r[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = unpack2<T>(gw[t]);
            r[t] = pack2<T>(f.x * cc[2 * t], f.y * cc[2 * t + 1]);
        }
        *reinterpret_cast<uint4 *>(dgate + o) = make_uint4(r[0], r[1], r[2], r[3]);
    }
}

}  // namespace

cudaError_t launch_gate_grad(const Prob &p, const void *dO, const float *c, void *dgate, cudaStream_t s) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long units = (long long)p.B * p.nQ * p.tile_q * p.Hq;
    const long long want = (units * 16 + 255) / 256;
    const int grid = (int)(want < (long long)sms * 8 ? (want < 1 ? 1 : want) : (long long)sms * 8);
    prof_begin("gate_grad", s);
    if (p.dtype == T_BF16)
        k_gate_grad<__nv_bfloat16><<<grid, 256, 0, s>>>(p, (const __nv_bfloat16 *)dO, c, (__nv_bfloat16 *)dgate);
    else
        k_gate_grad<__half><<<grid, 256, 0, s>>>(p, (const __half *)dO, c, (__half *)dgate);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const Prob &p, const void *dO, const void *o, const float *lse, float *nlse2,
                            float *ndvec, unsigned *err, cudaStream_t s) {
    const long long slots = (long long)p.B * p.Hq * p.nQ * p.tile_q;
    if (slots == 0) return cudaSuccess;
    if (slots > (long long)INT_MAX) return cudaErrorInvalidValue;
    CUtensorMap tdo, to;
    if (!make_tmap_rows(&tdo, p, true, dO, p.Hq, kPrepRows) || !make_tmap_rows(&to, p, true, o, p.Hq, kPrepRows))
        return cudaErrorInvalidValue;
    const int ntasks = (int)(slots / kPrepRows);  // tile_q is a multiple of 64
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = ntasks < sms ? ntasks : sms;  // one CTA per SM (the ring fills its shared memory)
    const cudaError_t ae = p.dtype == T_BF16
                               ? ensure_smem_limit((const void *)k_bwd_prep<__nv_bfloat16>, (int)kPrepSmem)
                               : ensure_smem_limit((const void *)k_bwd_prep<__half>, (int)kPrepSmem);
    if (ae != cudaSuccess) return ae;
    prof_begin("bwd_prep", s);
    if (p.dtype == T_BF16)
        k_bwd_prep<__nv_bfloat16><<<blocks, kPrepThreads, kPrepSmem, s>>>(tdo, to, p, lse, nlse2, ndvec, ntasks, err);
    else
        k_bwd_prep<__half><<<blocks, kPrepThreads, kPrepSmem, s>>>(tdo, to, p, lse, nlse2, ndvec, ntasks, err);
    prof_end(s);
    return cudaGetLastError();
}

long long dk_units(const Prob &p) { return (long long)p.B * p.Hkv * p.nKV * (p.tile_kv / 128); }

cudaError_t launch_dk_order(const Prob &p, const int *kv_ptr, int cap, int *order, int *keys, cudaStream_t s) {
    const long long units = dk_units(p);
    if (units == 0) return cudaSuccess;
    if (units > (long long)INT_MAX) return cudaErrorInvalidValue;
    prof_begin("dkdv_order", s);
    k_dk_order<<<p.B * p.Hkv, kOrderThreads, 0, s>>>(p, kv_ptr, cap, order, keys);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const Prob &p, const BwdArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv, tdo, tdk, tdv;
    if (!make_tmap_rows(&tq, p, true, a.q, p.Hq, kDkItem) || !make_tmap_rows(&tk, p, false, a.k, p.Hkv) ||
        !make_tmap_rows(&tv, p, false, a.v, p.Hkv) || !make_tmap_rows(&tdo, p, true, a.dO, p.Hq, kDkItem) ||
        !make_tmap_rows(&tdk, p, false, a.dk, p.Hkv) || !make_tmap_rows(&tdv, p, false, a.dv, p.Hkv))
        return cudaErrorInvalidValue;
    const long long units = dk_units(p);
    if (units == 0) return cudaSuccess;
    if (units > (long long)INT_MAX) return cudaErrorInvalidValue;
    dim3 grid((unsigned)units);
    const cudaError_t ae = p.dtype == T_BF16 ? ensure_smem_limit((const void *)k_dkdv<__nv_bfloat16>, (int)kDkSmem)
                                             : ensure_smem_limit((const void *)k_dkdv<__half>, (int)kDkSmem);
    if (ae != cudaSuccess) return ae;
    prof_begin("bwd_dkdv", s);
    if (p.dtype == T_BF16)
        k_dkdv<__nv_bfloat16><<<grid, kDkThreads, kDkSmem, s>>>(tq, tk, tv, tdo, tdk, tdv, p, a);
    else
        k_dkdv<__half><<<grid, kDkThreads, kDkSmem, s>>>(tq, tk, tv, tdo, tdk, tdv, p, a);
    prof_end(s);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const Prob &p, const BwdArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!make_tmap_rows(&tq, p, true, a.q, p.Hq) || !make_tmap_rows(&tk, p, false, a.k, p.Hkv) ||
        !make_tmap_rows(&tv, p, false, a.v, p.Hkv) || !make_tmap_rows(&tdo, p, true, a.dO, p.Hq) ||
        !make_tmap_rows(&tdq, p, true, a.dq, p.Hq))
        return cudaErrorInvalidValue;
    dim3 grid(p.nQ * (p.tile_q / 128), p.Hq, p.B);
    const cudaError_t ae = p.dtype == T_BF16 ? ensure_smem_limit((const void *)k_dq<__nv_bfloat16>, (int)kDqSmem)
                                             : ensure_smem_limit((const void *)k_dq<__half>, (int)kDqSmem);
    if (ae != cudaSuccess) return ae;
    prof_begin("bwd_dq", s);
    if (p.dtype == T_BF16)
        k_dq<__nv_bfloat16><<<grid, kDqThreads, kDqSmem, s>>>(tq, tk, tv, tdo, tdq, p, a);
    else
        k_dq<__half><<<grid, kDqThreads, kDqSmem, s>>>(tq, tk, tv, tdo, tdq, p, a);
    prof_end(s);
    return cudaGetLastError();
}


}  // namespace vsa
