// vsa_internal.h -- host-side declarations shared by the library's
// translation units (kernel launchers and the instrumentation hooks).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vsa.h"
#include "vsa_common.cuh"

namespace vsa {

// Instrumentation: every launcher brackets its kernel with these.
void prof_begin(const char *name, cudaStream_t s);
void prof_end(cudaStream_t s);
// VSA_OK for cudaSuccess; otherwise records the error (vsa_last_cuda_error)
// and returns VSA_ERR_CUDA.
vsa_status status_from_cuda(cudaError_t e);
// vsa_bwd_reuse that also records `dkdv_done` on the stream once dk and dv
// are final (after the dK/dV pass, before the dQ pass), so a caller can
// start copying them while dQ is computed.
vsa_status bwd_reuse_event(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                           const void *o_sparse, const float *lse, const int32_t *q_idx, const int32_t *q_cnt,
                           int idx_cap, const int32_t *kv_ptr, const int32_t *kv_qidx, const int32_t *q_var,
                           const int32_t *kv_var, const void *gate, void *dq, void *dk, void *dv, int reuse,
                           void *workspace, size_t workspace_bytes, vsa_stream_t stream, cudaEvent_t dkdv_done);

// Identity (cuCtxGetId) of the calling thread's current CUDA context, 0 if
// there is none yet. A device reset gives the device a new context and so
// a new id, which is how per-device set-up learns it must be redone.
unsigned long long current_context_id();
// Raises a kernel's dynamic shared-memory limit to at least `bytes` in the
// current context (the attribute belongs to the device's context, so every
// GPU and every context after a reset gets its own call); a later call with
// a larger size raises it again. Thread-safe.
cudaError_t ensure_smem_limit(const void *kernel, int bytes);

// Host-side validation shared by the entry points: descriptor -> Prob
// (VSA_OK or the status to return; scale 0 becomes 1/sqrt(D)); the tile
// fills become part of the Prob in the padded layouts (need_q: q_var is
// required too).
bool aligned16(const void *ptr);
vsa_status to_prob(const vsa_desc *d, Prob *p);
vsa_status need_vars(const Prob &p, const int32_t *q_var, const int32_t *kv_var, Prob *out, bool need_q);
// Every argument check of vsa_build_block_map except the workspace's.
vsa_status block_map_prob(const vsa_desc *desc, const void *q, const void *k, const int32_t *q_var,
                          const int32_t *kv_var, int topk, int need_bwd_index, const uint8_t *block_map,
                          const int32_t *q_idx, const int32_t *q_cnt, int idx_cap, const int32_t *kv_ptr,
                          const int32_t *kv_qidx, Prob *p);
// The block-map step's launches with the tile means in pq / pk.
vsa_status run_block_map(const Prob &p, const void *q, const void *k, int topk, int need_bwd_index,
                         uint8_t *block_map, int32_t *q_idx, int32_t *q_cnt, int idx_cap, int32_t *kv_ptr,
                         int32_t *kv_qidx, float *pq, float *pk, cudaStream_t s);

// Tile pooling (fp32 means of the first var tokens), [B, H, nT, D].
struct PoolSeg {
    const void *x;     // q, k or v in the problem's layout
    float *out;        // tile means [B, H, nT, D]
    int q_side;        // 1: query tiles (q_var), 0: key/value tiles (kv_var)
    long long warps;   // filled by launch_pools
};
struct PoolSegs {
    PoolSeg s[3];
    int n;
};
cudaError_t launch_pools(const Prob &p, const PoolSegs &segs, cudaStream_t s);
// Any of q, k, v in one launch; a NULL tensor is skipped (nothing launched
// when all three are NULL).
cudaError_t launch_pool_qkv(const Prob &p, const void *q, float *pq, const void *k, float *pk, const void *v,
                            float *pv, cudaStream_t s);
// Coarse scores + per-row top-k -> block map and Q-owned index.
cudaError_t launch_select(const Prob &p, const float *pq, const float *pk, int topk, uint8_t *map,
                          int *q_idx, int *q_cnt, int cap, cudaStream_t s);
// Caller-given block map -> Q-owned index.
cudaError_t launch_mask_index(const Prob &p, const uint8_t *map, int *q_idx, int *q_cnt, int cap,
                              cudaStream_t s);
// Query-block mask [B, Hq, nQb, nKV] (block_q rows per block) -> tile map
// (union over each tile's blocks), Q-owned index with per-entry block bit
// masks, and (kv_ptr != NULL) the KV-owned index with its bit masks.
cudaError_t launch_block_index(const Prob &p, int bq, int nQb, const uint8_t *bm, uint8_t *tmap, int *q_idx,
                               int *q_cnt, int *q_sub, int cap, int *kv_ptr, int *kv_qidx, int *kv_qsub,
                               cudaStream_t s);
// Block map -> KV-owned index.
cudaError_t launch_transpose(const Prob &p, const uint8_t *map, int *kv_ptr, int *kv_qidx, int cap,
                             cudaStream_t s);

// Largest nKV the selection kernel handles (its shared-memory score rows).
constexpr int kMaxSelectKV = 3072;
// Largest number of 128-key chunks one query tile may visit.
constexpr int kMaxChunks = 1024;

// Forward attention (tcgen05). out / o_sparse / gate / c as in vsa_fwd.
struct FwdArgs {
    const void *q, *k, *v;
    const int *q_idx, *q_cnt;
    int cap;
    void *out, *o_sparse;
    float *lse;
    const void *gate;   // NULL: no compression
    const float *c;     // [B, Hq, nQ, D] compression output (gate != NULL)
    const int *q_sub;   // per-entry query-block bit masks (NULL: whole tiles)
    int block_q;        // rows per query block when q_sub != NULL
    unsigned *err;
    uint8_t *redo;      // [B, Hq, nQ] tiles the CTA-pair kernel hands to the single-CTA one
    int redo_only;      // single-CTA kernel: compute only the tiles marked in redo
};
cudaError_t launch_fwd(const Prob &p, const FwdArgs &a, cudaStream_t s);

// Compression branch, forward: c_i = sum_j softmax_j(scale pq.pk_j) pv_j.
// Gated compression, gradient of the gate: dgate_t = dO_t (*) c_(tile of t).
cudaError_t launch_gate_grad(const Prob &p, const void *dO, const float *c, void *dgate, cudaStream_t s);
cudaError_t launch_compress_fwd(const Prob &p, const float *pq, const float *pk, const float *pv,
                                float *c, cudaStream_t s);

// Backward pieces.
// Backward preprocess: per query slot of the padded tile layout
// [B, Hq, nQ * tile_q], nlse2 = -LSE * log2(e) and ndvec = -Dvec with
// Dvec = dO . O, both negated so that P = 2^(scale log2e S + nlse2) and
// dP - Dvec = dP + ndvec are single adds (slots past a varlen sequence's
// end get nlse2 = -inf, ndvec = 0).
cudaError_t launch_bwd_prep(const Prob &p, const void *dO, const void *o, const float *lse, float *nlse2,
                            float *ndvec, unsigned *err, cudaStream_t s);
struct BwdArgs {
    const void *dO, *q, *k, *v;
    const float *nlse2, *ndvec;   // padded tile layout, see launch_bwd_prep
    const int *q_idx, *q_cnt;
    int cap;
    const int *kv_ptr, *kv_qidx;
    void *dq, *dk, *dv;
    const float *dpq, *dpk, *dpv;   // compression gradients (NULL without a gate)
    const int *q_sub, *kv_qsub;     // query-block bit masks of both indices (NULL: whole tiles)
    int block_q;
    unsigned *err;
    const int *dk_order;            // dK/dV units, longest work first (launch_dk_order)
};
// Units of the dK/dV pass: one per (batch entry, key/value head, 128-key
// chunk), numbered ((b * Hkv + hk) * nKV + j) * (tile_kv / 128) + chunk.
long long dk_units(const Prob &p);
// Writes order[dk_units], a permutation of the units: the (b, key/value
// head) segments in grid order, each segment's units by decreasing work
// (the summed KV-owned list lengths of the unit's GQA group, from kv_ptr);
// keys[dk_units] is scratch. One CTA per segment.
cudaError_t launch_dk_order(const Prob &p, const int *kv_ptr, int cap, int *order, int *keys, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const Prob &p, const BwdArgs &a, cudaStream_t s);
cudaError_t launch_bwd_dq(const Prob &p, const BwdArgs &a, cudaStream_t s);
// Compression branch, backward: dc, then A / ds per row, then the
// per-KV-tile column sums.
cudaError_t launch_compress_bwd(const Prob &p, const void *dO, const void *gate, const float *pq,
                                const float *pk, const float *pv, float *dc, float *A, float *ds,
                                float *dpq, float *dpk, float *dpv, cudaStream_t s);

// Tensor-map encoding (driver entry point fetched through the runtime):
// boxes of 64 head dims x box_rows tokens of one head, 128-byte swizzle.
bool make_tmap_rows(CUtensorMap *map, const Prob &p, bool q_side, const void *base, int heads,
                    int box_rows = 128);

}  // namespace vsa
