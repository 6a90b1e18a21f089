// check_inputs.cu -- vsa_check_inputs: an opt-in pass that validates the
// device-resident arguments the host checks cannot see (tile fills, varlen
// offsets and both block indices) before they reach the attention kernels.
//
// Pages: FastVideo block_sparse_attn_cute_fwd.py (_vbs_mask_mod: key n of a
// tile is valid iff n mod tile < vbs, which reads vbs as a count in
// [0, tile]; _map_to_index's rank and residency checks; the KV-owned
// backward index of _build_sparse_tensors lists, per KV tile, the query
// tiles that selected it); Ascend test_npu_block_sparse_attention_backward.py
// (actual_seq_lengths: per-sequence lengths of the TND layout, cumulative).
//
// Every kernel here reads only inside the buffers the declared sizes give
// (nQ, nKV, B + 1 offsets, B*Hq*nQ counts of at most idx_cap entries,
// B*Hq*(nKV+1) offsets and B*Hq*nQ*idx_cap entries) and never dereferences
// a value it is checking. A failed check records its code in the status
// word (the first failure wins) and nothing else.
#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

enum : unsigned {
    kBadQVar = 0xC001,       // q_var[i] outside [0, tile_q]
    kBadKvVar = 0xC002,      // kv_var[j] outside [0, tile_kv]
    kBadCuQ = 0xC003,        // cu_seqlens_q negative, decreasing, past T_q, or a sequence longer than nQ tiles
    kBadCuKv = 0xC004,       // the same for cu_seqlens_kv
    kBadQCnt = 0xC005,       // q_cnt outside [0, idx_cap]
    kBadQIdx = 0xC006,       // q_idx entry outside [0, nKV), not ascending, or a tile without valid tokens
    kBadKvPtr = 0xC007,      // kv_ptr[0] != 0, decreasing, or past nQ * idx_cap
    kBadKvQidx = 0xC008,     // kv_qidx entry outside [0, nQ) or not ascending within its KV tile
    kNotTranspose = 0xC009,  // the KV-owned index is not the transpose of the Q-owned one
};

__device__ __forceinline__ void flag(unsigned *err, bool bad, unsigned code) {
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_error(err, code);
}

// Tile fills (padded layouts) or sequence offsets (TND); one block.
__global__ void __launch_bounds__(256) k_check_fill(Prob p, const int *q_var, const int *kv_var, unsigned *err) {
    if (p.layout != L_TND) {
        for (int i0 = 0; i0 < p.nQ; i0 += blockDim.x) {
            const int i = i0 + threadIdx.x;
            flag(err, i < p.nQ && (q_var[i] < 0 || q_var[i] > p.tile_q), kBadQVar);
        }
        for (int j0 = 0; j0 < p.nKV; j0 += blockDim.x) {
            const int j = j0 + threadIdx.x;
            flag(err, j < p.nKV && (kv_var[j] < 0 || kv_var[j] > p.tile_kv), kBadKvVar);
        }
        return;
    }
    for (int side = 0; side < 2; ++side) {
        const int *cu = side == 0 ? p.cu_q : p.cu_kv;
        const long long total = side == 0 ? p.Sq : p.Skv;
        const long long longest = side == 0 ? (long long)p.nQ * p.tile_q : (long long)p.nKV * p.tile_kv;
        for (int b0 = 0; b0 <= p.B; b0 += blockDim.x) {
            const int b = b0 + threadIdx.x;
            bool bad = false;
            if (b <= p.B) {
                const long long c = cu[b];
                bad = c < 0 || c > total;
                if (b > 0) {
                    const long long len = c - cu[b - 1];
                    bad = bad || len < 0 || len > longest;
                }
            }
            flag(err, bad, side == 0 ? kBadCuQ : kBadCuKv);
        }
    }
}

// Q-owned index: one warp per (b, h, query tile).
__global__ void __launch_bounds__(256) k_check_qidx(Prob p, const int *q_idx, const int *q_cnt, int cap,
                                                    unsigned *err) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= (long long)p.B * p.Hq * p.nQ) return;
    const int lane = threadIdx.x & 31;
    const int b = (int)(row / ((long long)p.Hq * p.nQ));
    const int cnt = q_cnt[row];
    if (cnt < 0 || cnt > cap) {
        if (lane == 0) set_error(err, kBadQCnt);
        return;
    }
    const int *idx = q_idx + row * cap;
    for (int n0 = 0; n0 < cnt; n0 += 32) {
        const int n = n0 + lane;
        bool bad = false;
        if (n < cnt) {
            const int j = idx[n];
            bad = j < 0 || j >= p.nKV || (n > 0 && idx[n - 1] >= j);
            bad = bad || kv_valid(p, b, j) == 0;
        }
        flag(err, bad, kBadQIdx);
    }
}

// KV-owned index of one (b, h): one block. Offsets must start at 0, never
// decrease and stay within nQ * cap; entries lie in [0, nQ) and ascend
// within each KV tile. With the Q-owned index given, every entry (i of KV
// tile j) must appear in query tile i's list and the entry count must equal
// the Q-owned lists' total, which together make the two indices transposes
// of each other (both are duplicate-free).
__global__ void __launch_bounds__(256) k_check_kvidx(Prob p, const int *kv_ptr, const int *kv_qidx,
                                                     const int *q_idx, const int *q_cnt, int cap, unsigned *err) {
    __shared__ int s_bad;
    __shared__ int s_sum[8];
    const long long bh = (long long)blockIdx.y * p.Hq + blockIdx.x;
    const int *ptr = kv_ptr + bh * (p.nKV + 1);
    const int *lst = kv_qidx + bh * (long long)p.nQ * cap;
    const int cap_all = p.nQ * cap;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int j = threadIdx.x; j <= p.nKV; j += blockDim.x) {
        const int v = ptr[j];
        const bool bad = (j == 0 && v != 0) || (j > 0 && v < ptr[j - 1]) || v < 0 || v > cap_all;
        if (bad) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) set_error(err, kBadKvPtr);
        return;
    }
    const int total = ptr[p.nKV];
    if (q_idx) {
        int sum = 0;
        for (int i = threadIdx.x; i < p.nQ; i += blockDim.x) sum += clampi(q_cnt[bh * p.nQ + i], 0, cap);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if ((threadIdx.x & 31) == 0) s_sum[threadIdx.x >> 5] = sum;
        __syncthreads();
        if (threadIdx.x == 0) {
            int all = 0;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) all += s_sum[w];
            if (all != total) set_error(err, kNotTranspose);
        }
    }
    for (int pos = threadIdx.x; pos < total; pos += blockDim.x) {
        int lo = 0, hi = p.nKV;  // the KV tile whose list holds pos: largest j with ptr[j] <= pos
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (ptr[mid] <= pos) lo = mid; else hi = mid;
        }
        const int j = lo, i = lst[pos];
        if (i < 0 || i >= p.nQ || (pos > ptr[j] && lst[pos - 1] >= i)) {
            set_error(err, kBadKvQidx);
            continue;
        }
        if (q_idx) {
            const long long row = bh * p.nQ + i;
            const int *qi = q_idx + row * cap;
            int a = 0, c = clampi(q_cnt[row], 0, cap);  // binary search for j in the ascending list
            while (a < c) {
                const int mid = (a + c) >> 1;
                if (qi[mid] < j) a = mid + 1; else c = mid;
            }
            if (a >= clampi(q_cnt[row], 0, cap) || qi[a] != j) set_error(err, kNotTranspose);
        }
    }
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" vsa_status vsa_check_inputs(const vsa_desc *desc, const int32_t *q_var, const int32_t *kv_var,
                                       const int32_t *q_idx, const int32_t *q_cnt, int idx_cap,
                                       const int32_t *kv_ptr, const int32_t *kv_qidx, void *workspace,
                                       size_t workspace_bytes, vsa_stream_t stream, int32_t *code) {
    Prob p0, p;
    vsa_status st = to_prob(desc, &p0);
    if (st != VSA_OK) return st;
    if ((st = need_vars(p0, q_var, kv_var, &p, true)) != VSA_OK) return st;
    if (!code) return VSA_ERR_NULL;
    if (!q_idx != !q_cnt || !kv_ptr != !kv_qidx) return VSA_ERR_NULL;  // each index whole or absent
    if ((q_idx || kv_ptr) && (idx_cap < 1 || idx_cap > p.nKV)) return VSA_ERR_SHAPE;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < 256)
        return VSA_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *err = static_cast<unsigned *>(workspace);
    prof_begin("check_fill", s);
    k_check_fill<<<1, 256, 0, s>>>(p, p.q_var, p.kv_var, err);
    prof_end(s);
    cudaError_t e = cudaGetLastError();
    const long long rows = (long long)p.B * p.Hq * p.nQ;
    if (e == cudaSuccess && q_idx) {
        prof_begin("check_qidx", s);
        k_check_qidx<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, q_idx, q_cnt, idx_cap, err);
        prof_end(s);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && kv_ptr) {
        prof_begin("check_kvidx", s);
        k_check_kvidx<<<dim3(p.Hq, p.B), 256, 0, s>>>(p, kv_ptr, kv_qidx, q_idx, q_cnt, idx_cap, err);
        prof_end(s);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return status_from_cuda(e);
    st = vsa_device_status(workspace, stream, code);
    if (st == VSA_ERR_DEVICE && (*code & 0xFF00) == 0xC000) return VSA_ERR_SHAPE;
    return st;
}
