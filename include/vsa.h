/*
 * vsa.h -- C ABI of the GB300 (sm_103a) tile-top-k block-sparse video
 * attention library (libvsa.so): forward and backward of softmax attention
 * restricted, per query tile, to the key/value tiles chosen by top-k over
 * tile-mean-pooled ("coarse") scores, with per-tile valid-token counts that
 * trim padded 3D video tiles, and an optional gated compression branch.
 *
 * Sources (page titles, with the section that defines each operation):
 *   [VSA-test]  FastVideo fastvideo-kernel/tests/test_vsa256_backward.py
 *   [FA4-adapt] FastVideo fastvideo-kernel/python/fastvideo_kernel/
 *               block_sparse_attn_cute_fwd.py
 *   [NPU-test]  Ascend op-plugin test/test_custom_ops/
 *               test_npu_block_sparse_attention_backward.py
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers on the current CUDA device,
 *   owned by the caller. The library allocates no device memory, frees
 *   nothing and never synchronises: each call validates its arguments on
 *   the host, enqueues kernels on `stream` and returns. Outputs are
 *   overwritten, never accumulated into.
 * - q, dO, out, o_sparse, gate and dq share the layout `layout` with Hq
 *   heads; k, v, dk and dv share it with Hkv heads (GQA: query head h reads
 *   key/value head h / (Hq / Hkv), as in [NPU-test]
 *   cpu_block_sparse_attention_tnd_gqa_with_lse). All are dense (the last
 *   dimension D is contiguous, no gaps) and 16-byte aligned.
 *     VSA_LAYOUT_BHSD  [B, H, S, D]
 *     VSA_LAYOUT_BSHD  [B, S, H, D]
 *     VSA_LAYOUT_TND   [T, H, D], sequences packed along T with device
 *                      offsets cu_seqlens_* ([B+1] int32, ascending).
 * - In the padded video layouts each batch entry holds nQ query tiles of
 *   tile_q tokens and nKV key/value tiles of tile_kv tokens; the first
 *   q_var[i] / kv_var[j] slots of a tile are its valid tokens and the rest
 *   are zero padding ([VSA-test] _zero_pad_tail). q_var / kv_var are device
 *   int32 arrays [nQ] / [nKV], shared by every batch entry and head, each
 *   value in [0, tile] ([FA4-adapt] _vbs_mask_mod reads it as a count of
 *   valid slots). In TND the valid tokens of tile t of sequence b are
 *   min(tile, len_b - t*tile) (zero past the end) and q_var / kv_var are
 *   ignored (pass NULL).
 * - Device-resident arguments (tile fills, cu_seqlens_*, the two block
 *   indices) cannot be checked on the host without a synchronisation, so
 *   the calls below do not check them; vsa_check_inputs does, on request.
 *   Given values outside their ranges anyway, the kernels still read and
 *   write only inside the caller's buffers (fills, offsets, counts and
 *   entries are clamped into range), but the results are meaningless.
 * - Every query slot of a padded Q tile is a query row (the valid-length
 *   mask applies to keys only, [FA4-adapt] _vbs_mask_mod); in TND only
 *   rows inside a sequence exist and only those are written.
 * - The LSE is fp32, natural log, head-major: [B, Hq, Sq] for the padded
 *   layouts and [Hq, T] for TND ([VSA-test] test_vsa256_cute_lse_is_bhs).
 *   A row whose selected tiles hold no valid key gets O = 0, LSE = -inf.
 * - Block index (Q-owned CSR): q_idx [B, Hq, nQ, idx_cap] int32 lists, per
 *   query tile, the selected KV tiles that hold at least one valid token,
 *   ascending; q_cnt [B, Hq, nQ] counts them; unused slots are -1.
 * - Transposed index (KV-owned CSR, one per query head): kv_ptr
 *   [B, Hq, nKV+1] int32 offsets into kv_qidx [B, Hq, nQ*idx_cap], which
 *   lists, for KV tile j, the query tiles whose index holds j, ascending
 *   ([FA4-adapt] _build_sparse_tensors, KV-owned backward metadata).
 *   Entries past kv_ptr[nKV] are -1.
 * - workspace is caller-allocated device scratch of at least
 *   vsa_workspace_size() bytes, 256-byte aligned. Its first 256 bytes hold
 *   a device status word that kernels set if an internal wait times out
 *   (read it with vsa_device_status). The rest is scratch; the only values
 *   one call passes to the next are the tile means that vsa_fwd_reuse /
 *   vsa_bwd_reuse are told to keep. Calls that share a workspace must not
 *   run concurrently.
 */
#ifndef VSA_H
#define VSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *vsa_stream_t; /* same type as cudaStream_t */

typedef enum {
    VSA_OK = 0,
    VSA_ERR_NULL = 1,            /* a required pointer is NULL */
    VSA_ERR_SHAPE = 2,           /* sizes inconsistent, idx_cap too small; vsa_check_inputs: a fill,
                                    offset or index entry out of range */
    VSA_ERR_DTYPE = 3,           /* dtype not bf16 / fp16 */
    VSA_ERR_LAYOUT = 4,          /* unknown layout, or a pointer not 16-byte aligned */
    VSA_ERR_UNSUPPORTED = 5,     /* D != 128, tile not 128/256, or a size past a kernel limit */
    VSA_ERR_MISSING_SEQLENS = 6, /* TND without both cu_seqlens_q and cu_seqlens_kv */
    VSA_ERR_WORKSPACE = 7,       /* workspace NULL, misaligned or smaller than required */
    VSA_ERR_CUDA = 8,            /* a CUDA runtime call or kernel launch failed */
    VSA_ERR_DEVICE = 9,          /* a kernel recorded a failed internal wait (see vsa_device_status) */
    VSA_ERR_SCRATCH = 10         /* problem too large for vsa_build_block_map_static's fixed scratch */
} vsa_status;

typedef enum { VSA_LAYOUT_BHSD = 0, VSA_LAYOUT_BSHD = 1, VSA_LAYOUT_TND = 2 } vsa_layout;
typedef enum { VSA_DTYPE_BF16 = 0, VSA_DTYPE_FP16 = 1 } vsa_dtype;

/* Problem descriptor (host memory; pointed-to seqlens are device memory). */
typedef struct {
    int32_t layout;     /* vsa_layout */
    int32_t dtype;      /* vsa_dtype of q, k, v, dO, gate, out, o_sparse, dq, dk, dv */
    int32_t B;          /* batch entries (TND: number of sequences) */
    int32_t Hq, Hkv;    /* query heads, key/value heads; Hq % Hkv == 0 */
    int32_t D;          /* head dim; must be 128 */
    int32_t Sq, Skv;    /* padded layouts: tokens per batch entry, = nQ*tile_q and
                           nKV*tile_kv. TND: total tokens T_q, T_kv */
    int32_t tile_q;     /* tokens per query tile: 128 or 256 */
    int32_t tile_kv;    /* tokens per key/value tile: 128 or 256 */
    int32_t nQ, nKV;    /* tiles per batch entry. TND: ceil(max_len / tile) */
    const int32_t *cu_seqlens_q;  /* TND only: device [B+1] token offsets */
    const int32_t *cu_seqlens_kv; /* TND only: device [B+1] token offsets */
    float scale;        /* softmax scale on q.k; 0 means 1/sqrt(D) */
} vsa_desc;

/* Bytes of workspace needed by every call below for this problem (with or
 * without the gated compression branch). */
size_t vsa_workspace_size(const vsa_desc *desc, int with_gate);

/* Block-map step. Tile means of q (over the first q_var[i] tokens, per
 * query head) and of k (first kv_var[j] tokens, per key/value head) in
 * fp32, a sequential round-to-nearest sum then an IEEE divide; raw coarse
 * scores r_ij = pq_i . pk_j as an fp32 fma chain over ascending d; per
 * query tile, the min(topk, nKV) largest r_ij under (r desc, j asc), with
 * r = -inf for tiles without valid tokens. The pages call the step with
 * (q, k, q_var, kv_var, topk) ([VSA-test] video_sparse_attn's topk argument;
 * [FA4-adapt] _map_to_index and the vbs > 0 split for the index).
 * Writes block_map [B, Hq, nQ, nKV] uint8 (1 = selected), q_idx / q_cnt
 * (idx_cap >= min(topk, nKV)) and, when need_bwd_index != 0, the
 * transposed index kv_ptr / kv_qidx; with need_bwd_index == 0 those two may
 * be NULL and are not touched (the inference fast path of [FA4-adapt]
 * _build_sparse_tensors). The result is bit-identical across runs and
 * independent of need_bwd_index. In TND a query tile past its sequence's
 * end selects nothing. */
vsa_status vsa_build_block_map(const vsa_desc *desc, const void *q, const void *k,
                               const int32_t *q_var, const int32_t *kv_var, int topk,
                               int need_bwd_index, uint8_t *block_map, int32_t *q_idx,
                               int32_t *q_cnt, int idx_cap, int32_t *kv_ptr, int32_t *kv_qidx,
                               void *workspace, size_t workspace_bytes, vsa_stream_t stream);

/* vsa_build_block_map for callers that cannot allocate device memory.
 * The pages have no counterpart. It exists for callers that may not call
 * cudaMalloc at all: a runtime or memory pool that owns every byte of the
 * device and has no workspace to lend, an allocator that forbids outside
 * allocations, or code on a path where an allocation could synchronise the
 * device or fail. Same arguments, checks, results and errors as
 * vsa_build_block_map (the same validation and launches run), minus the
 * workspace: the scratch for the fp32 tile means lives in a fixed array
 * inside libvsa.so (16 MiB, 4,194,304 floats, held on every GPU that loads
 * the library until the process exits). A problem needs B*Hq*nQ*128 +
 * B*Hkv*nKV*128 floats of it (plus alignment padding of at most 63
 * floats); larger problems return VSA_ERR_SCRATCH before anything is
 * launched. No cudaMalloc, cudaFree or allocating library routine is
 * called. The first call on a device (and the first after a device reset)
 * looks up the array's device address with that device current
 * (cudaGetSymbolAddress) and keeps it; make that first call before any
 * stream capture. Every call shares the one array, which keeps the last
 * call's contents: calls whose kernels may overlap on the GPU (different
 * streams, or several host threads) race on it and must be serialised by
 * the caller. Nothing in the array needs clearing between calls: each call
 * writes every element it later reads. */
vsa_status vsa_build_block_map_static(const vsa_desc *desc, const void *q, const void *k,
                                      const int32_t *q_var, const int32_t *kv_var, int topk,
                                      int need_bwd_index, uint8_t *block_map, int32_t *q_idx,
                                      int32_t *q_cnt, int idx_cap, int32_t *kv_ptr, int32_t *kv_qidx,
                                      vsa_stream_t stream);

/* Index step for a caller-given block map [B, Hq, nQ, nKV] uint8 (nonzero
 * = attend), as in [NPU-test] (block_sparse_mask) and [FA4-adapt]
 * _map_to_index. Tiles without valid tokens, and in TND blocks past either
 * sequence's end, are dropped. idx_cap >= nKV. kv_ptr / kv_qidx as for
 * vsa_build_block_map. */
vsa_status vsa_mask_to_index(const vsa_desc *desc, const uint8_t *block_map,
                             const int32_t *q_var, const int32_t *kv_var, int need_bwd_index,
                             int32_t *q_idx, int32_t *q_cnt, int idx_cap, int32_t *kv_ptr,
                             int32_t *kv_qidx, vsa_stream_t stream);

/* Forward. For every query row t of query tile i: softmax over the valid
 * keys of the KV tiles in q_idx[.., i, :] of scale * q_t . k_u, O_t =
 * sum_u P_tu v_u, LSE_t = max + ln(sum exp(s - max)) ([NPU-test]
 * cpu_block_sparse_attention_tnd_gqa_with_lse with the key mask of
 * [FA4-adapt] _vbs_mask_mod). Writes o_sparse (the attention output) and
 * lse. With gate == NULL, out receives O as well (o_sparse may then be
 * NULL or equal to out). With a gate (q-shaped, elementwise), the gated
 * compression branch adds, on every query row of tile i,
 * out_t = O_t + gate_t (*) c_i, c_i = sum_j softmax_j(scale pq_i . pk_j) pv_j
 * over the non-empty KV tiles, from the tile means of q, k, v ([VSA-test]
 * test_vsa256_cute_backward_with_compress_gate); o_sparse must then be a
 * separate buffer (the composition never overwrites the sparse output). */
vsa_status vsa_fwd(const vsa_desc *desc, const void *q, const void *k, const void *v,
                   const int32_t *q_idx, const int32_t *q_cnt, int idx_cap,
                   const int32_t *q_var, const int32_t *kv_var, const void *gate, void *out,
                   float *lse, void *o_sparse, void *workspace, size_t workspace_bytes,
                   vsa_stream_t stream);

/* Backward of vsa_fwd with the block index held fixed. Dvec_t = dO_t .
 * O_t (o_sparse); P = exp(scale q.k - LSE); dS = P (dO.v - Dvec);
 * dQ = scale sum dS k (Q-owned pass over q_idx); dK = scale sum dS^T q and
 * dV = sum P^T dO (KV-owned pass over kv_ptr / kv_qidx, summed over each
 * GQA group, no atomics) ([NPU-test] _softmax_backward_np and
 * cpu_block_sparse_attention_backward_tnd_gqa; [FA4-adapt]
 * _CuteAttentionQ128.backward). With a gate, the compression branch's
 * gradients flow to q, k, v through the tile means (1/var on the valid
 * slots); the gate receives none. dq has q's shape; dk, dv have k's.
 * Padded key slots get dk = dv = 0. */
vsa_status vsa_bwd(const vsa_desc *desc, const void *dO, const void *q, const void *k,
                   const void *v, const void *o_sparse, const float *lse, const int32_t *q_idx,
                   const int32_t *q_cnt, int idx_cap, const int32_t *kv_ptr,
                   const int32_t *kv_qidx, const int32_t *q_var, const int32_t *kv_var,
                   const void *gate, void *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, vsa_stream_t stream);

/* Tile means kept between the calls of one step. The gated compression
 * branch ([VSA-test] test_vsa256_cute_backward_with_compress_gate) reads
 * the fp32 tile means of q, k and v, and the block map already computed
 * those of q and k; vsa_fwd and vsa_bwd recompute every mean they read.
 * vsa_fwd_reuse / vsa_bwd_reuse are the same calls with a `reuse` mask
 * that names the means the workspace already holds for this call's inputs,
 * which are then read from it instead of recomputed (the pooling kernel
 * skips them; with every mean kept it is not launched):
 *   VSA_REUSE_QK_MEANS  pq, pk: the last vsa_build_block_map, vsa_fwd* or
 *                       vsa_bwd* run on this workspace had the same
 *                       descriptor, q, k, q_var and kv_var, unchanged since;
 *   VSA_REUSE_V_MEANS   pv: the last gated vsa_fwd* or vsa_bwd* run on this
 *                       workspace had the same v and kv_var, unchanged since.
 * The means are computed by one kernel in a fixed order, so a kept mean is
 * bit-identical to a recomputed one and the results do not depend on the
 * mask. The library cannot check the claim: a mask that names means the
 * workspace does not hold gives results computed from stale means (no
 * error). Without a gate the mask has no effect. Bits other than these two
 * give VSA_ERR_SHAPE. reuse = 0 is vsa_fwd / vsa_bwd exactly. */
enum { VSA_REUSE_QK_MEANS = 1, VSA_REUSE_V_MEANS = 2 };
vsa_status vsa_fwd_reuse(const vsa_desc *desc, const void *q, const void *k, const void *v,
                         const int32_t *q_idx, const int32_t *q_cnt, int idx_cap,
                         const int32_t *q_var, const int32_t *kv_var, const void *gate, void *out,
                         float *lse, void *o_sparse, int reuse, void *workspace,
                         size_t workspace_bytes, vsa_stream_t stream);
vsa_status vsa_bwd_reuse(const vsa_desc *desc, const void *dO, const void *q, const void *k,
                         const void *v, const void *o_sparse, const float *lse,
                         const int32_t *q_idx, const int32_t *q_cnt, int idx_cap,
                         const int32_t *kv_ptr, const int32_t *kv_qidx, const int32_t *q_var,
                         const int32_t *kv_var, const void *gate, void *dq, void *dk, void *dv,
                         int reuse, void *workspace, size_t workspace_bytes,
                         vsa_stream_t stream);

/* Failure-path check: launches one warp that waits, with the library's
 * bounded mbarrier wait, on a barrier that nothing ever arrives on. After
 * limit_ns of wall time (0 < limit_ns <= 10 s) the wait gives up, records
 * its site code (0x7E57) in workspace's status word -- read and cleared by
 * vsa_device_status, exactly as a timed-out wait inside an attention
 * kernel -- and the kernel returns; the context stays usable. *completed
 * (device int32) receives 0 (timed out) or 1 (the wait returned as if the
 * phase had completed, a library defect). workspace: 256-byte aligned, at
 * least 256 bytes. */
vsa_status vsa_check_wait_timeout(void *workspace, unsigned long long limit_ns, int32_t *completed,
                                  vsa_stream_t stream);

/* Query blocks smaller than a tile ([NPU-test]: block_shape [32, 128] and
 * [64, 128] with an explicit block_sparse_mask): a caller's mask
 * block_mask [B, Hq, nQb, nKV] uint8 (nonzero = attend) whose rows are
 * query blocks of block_q rows (block_q a multiple of 32 dividing tile_q;
 * nQb <= nQ * tile_q / block_q; TND: per sequence, ceil(max_len /
 * block_q) blocks, blocks past a sequence's end ignored) and whose columns
 * are the KV tiles. The kernels keep tiles of tile_q query rows: a tile's
 * index lists the union of its blocks' selections, and q_sub [B, Hq, nQ,
 * idx_cap] int32 (bit s set iff block s of the tile selected the entry's
 * KV tile) and kv_qsub [B, Hq, nQ*idx_cap] (the same bits for the KV-owned
 * entries) mask the keys of the other blocks' rows. Outputs as for
 * vsa_mask_to_index plus tile_map [B, Hq, nQ, nKV] uint8 (the union map).
 * A row whose block selects nothing gets O = 0, LSE = -inf and no
 * gradient. vsa_fwd_blocks / vsa_bwd_blocks are vsa_fwd / vsa_bwd (no
 * compression branch) with these masks; block_q must equal the one the
 * index was built with. */
vsa_status vsa_mask_to_index_blocks(const vsa_desc *desc, int block_q, int nQb, const uint8_t *block_mask,
                                    const int32_t *q_var, const int32_t *kv_var, int need_bwd_index,
                                    uint8_t *tile_map, int32_t *q_idx, int32_t *q_cnt, int32_t *q_sub,
                                    int idx_cap, int32_t *kv_ptr, int32_t *kv_qidx, int32_t *kv_qsub,
                                    vsa_stream_t stream);
vsa_status vsa_fwd_blocks(const vsa_desc *desc, int block_q, const void *q, const void *k, const void *v,
                          const int32_t *q_idx, const int32_t *q_cnt, const int32_t *q_sub, int idx_cap,
                          const int32_t *q_var, const int32_t *kv_var, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, vsa_stream_t stream);
vsa_status vsa_bwd_blocks(const vsa_desc *desc, int block_q, const void *dO, const void *q, const void *k,
                          const void *v, const void *out, const float *lse, const int32_t *q_idx,
                          const int32_t *q_cnt, const int32_t *q_sub, int idx_cap, const int32_t *kv_ptr,
                          const int32_t *kv_qidx, const int32_t *kv_qsub, const int32_t *q_var,
                          const int32_t *kv_var, void *dq, void *dk, void *dv, void *workspace,
                          size_t workspace_bytes, vsa_stream_t stream);

/* Gradient of the compression gate (the pages' gate carries no gradient:
 * [VSA-test] builds it without requires_grad). With out = O + gate (*) c
 * (vsa_fwd, gated), dgate_t = dO_t (*) c_i for every slot t of query tile
 * i (TND: every row inside a sequence); c is recomputed from q, k, v.
 * dO and dgate are q-shaped in `layout` (dgate: same dtype), 16-byte
 * aligned; workspace sized by vsa_workspace_size(desc, 1). Errors as for
 * vsa_fwd. */
vsa_status vsa_gate_grad(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                         const int32_t *q_var, const int32_t *kv_var, void *dgate, void *workspace,
                         size_t workspace_bytes, vsa_stream_t stream);

/* 3D video tiling, the layout step on either side of the attention
 * ([VSA-test]: _BLOCK_SIZE_3D = (4, 8, 8), and _zero_pad_tail, by which
 * callers scatter a latent into a zeroed tile buffer so that the first var
 * slots of a tile are its tokens). The pages do not fix the orders; here
 * tiles are numbered in raster order of their (T, H, W) tile coordinates
 * and the tokens of a tile fill its first slots in raster order of its own
 * box, clipped at the latent's edges, so tile k holds var_k = product of
 * its clipped extents tokens, followed by zero slots.
 *   latent: device [B, T, H, W, row] with row = row_bytes bytes per token
 *           (e.g. heads x head_dim 16-bit values), dense;
 *   tiled:  device [B, nTiles * tT*tH*tW, row], i.e. BSHD with
 *           S = nTiles * tile (nTiles = vsa_tile_3d_count(...)).
 * Both pointers 16-byte aligned, row_bytes a multiple of 16; the two
 * buffers must not overlap. vsa_tile_3d writes every slot of `tiled`
 * (padding as zeros) and, if tile_var != NULL, the per-tile valid counts
 * tile_var[nTiles] (int32, device; the kv_var / q_var of the attention
 * calls). vsa_untile_3d writes every token of `latent` from the valid slots
 * of `tiled` and reads no padding slot. Errors: VSA_ERR_NULL, VSA_ERR_LAYOUT
 * (misaligned), VSA_ERR_SHAPE (non-positive size, row_bytes not a multiple
 * of 16), VSA_ERR_UNSUPPORTED (more than 2^31 - 1 slots), VSA_ERR_CUDA. */
int vsa_tile_3d_count(int T, int H, int W, int tT, int tH, int tW);
vsa_status vsa_tile_3d(int B, int T, int H, int W, int row_bytes, int tT, int tH, int tW,
                       const void *latent, void *tiled, int32_t *tile_var, vsa_stream_t stream);
vsa_status vsa_untile_3d(int B, int T, int H, int W, int row_bytes, int tT, int tH, int tW,
                         const void *tiled, void *latent, vsa_stream_t stream);

/* Head slices: every (batch, head) is an independent problem (the
 * per-(batch, head) loops of [NPU-test]'s TND/GQA golden, with key/value
 * head h / (Hq / Hkv) for query head h), so one problem's heads can be cut
 * into `groups` equal slices, each with Hq/groups query heads and
 * Hkv/groups key/value heads (Hkv % groups == 0, so every GQA group stays
 * whole inside one slice). Slice g (0 <= g < groups) holds query heads
 * [*q_head0, *q_head0 + slice->Hq) and key/value heads [*kv_head0,
 * *kv_head0 + slice->Hkv); *slice is desc with those head counts. Running
 * the calls above on each slice's tensors (the head slices of q, k, v, dO
 * and of every output, LSE and block index included) gives results
 * bit-identical to the whole problem's; this is how the host-buffer steps
 * below pipeline a problem and how a problem is split over GPUs with no
 * exchange between them. Host-only (no CUDA call). Errors: VSA_ERR_NULL,
 * the descriptor errors of the other calls, VSA_ERR_SHAPE for groups < 1,
 * Hkv % groups != 0 or g outside [0, groups). */
vsa_status vsa_head_slice(const vsa_desc *desc, int groups, int g, vsa_desc *slice, int32_t *q_head0,
                          int32_t *kv_head0);

/* One training step (block map, forward, backward; with gate != NULL also
 * the gated compression branch) from HOST buffers, with the copies
 * overlapped with the kernels. Every head is an independent problem (the
 * per-(batch, head) loops of [NPU-test]'s TND/GQA golden), so the heads are
 * cut into `groups` slices of Hq/groups query and Hkv/groups key/value
 * heads (Hkv % groups == 0; GQA groups stay whole). Slice g's inputs are
 * copied host -> device (strided 2D copies into a compact staging slot) on
 * an internal stream while earlier slices compute on `stream`, and each
 * slice's results are copied device -> host on a second internal stream as
 * soon as they are final (O and LSE after the forward, dk and dv after the
 * dK/dV pass, dq after the dQ pass); two staging slots alternate.
 * Each slice runs vsa_build_block_map (topk, with the KV-owned index),
 * vsa_fwd_reuse and vsa_bwd_reuse (the tile means pooled once per slice)
 * on its own descriptor, so every output is bit-identical to vsa_fwd and
 * vsa_bwd on the whole problem.
 *   q, k, v, dO:   host, in desc's layout and dtype (page-locked memory
 *                  lets the copies run asynchronously and overlap);
 *   gate:          host, q-shaped, or NULL (no compression branch); with a
 *                  gate, out = O + gate (*) c as in vsa_fwd, and the
 *                  backward's compression gradients are included;
 *   out, lse:      host outputs O and LSE (lse: fp32 [B, Hq, Sq], TND
 *                  [Hq, T_q]); either may be NULL (then not copied back);
 *   dq, dk, dv:    host gradients, shaped like q, k, v;
 *   q_var, kv_var, desc->cu_seqlens_*: device, as for the other calls;
 *   device_buf:    device staging memory (zeroed before its first use,
 *                  see vsa_step_host_status), 256-byte aligned, at least
 *                  vsa_train_step_host_size(desc, groups, topk,
 *                  gate != NULL) bytes (two slots of one slice's tensors,
 *                  indices, LSE and workspace), owned by the caller.
 * The call only enqueues work: everything it does is ordered after the
 * work already queued on `stream`, and `stream` reaches the end of the call
 * only after the last copy back has finished (synchronise `stream` before
 * reading the host outputs; keep the host buffers alive until then).
 * Errors: those of the three calls; VSA_ERR_SHAPE for groups < 1 or not
 * dividing Hkv, topk < 1; VSA_ERR_NULL for a missing required host
 * pointer; VSA_ERR_WORKSPACE for a NULL, misaligned or small device_buf;
 * VSA_ERR_CUDA when a copy, stream or event call fails.
 * vsa_train_step_host_size returns 0 for an invalid descriptor, groups or
 * topk. */
size_t vsa_train_step_host_size(const vsa_desc *desc, int groups, int topk, int with_gate);
vsa_status vsa_train_step_host(const vsa_desc *desc, int groups, const void *q, const void *k, const void *v,
                               const void *dO, const void *gate, const int32_t *q_var, const int32_t *kv_var,
                               int topk, void *out, float *lse, void *dq, void *dk, void *dv, void *device_buf,
                               size_t device_bytes, vsa_stream_t stream);

/* The same pipeline for inference: per head slice, vsa_build_block_map
 * (need_bwd_index = 0, the inference path of [FA4-adapt]
 * _build_sparse_tensors) and vsa_fwd (gated when gate != NULL), with q, k,
 * v (and gate) copied in and out (required) and lse (optional) copied back.
 * device_buf as for vsa_train_step_host (vsa_train_step_host_size covers
 * this call too). Errors as for vsa_train_step_host; VSA_ERR_NULL also
 * when out is NULL. */
vsa_status vsa_fwd_step_host(const vsa_desc *desc, int groups, const void *q, const void *k, const void *v,
                             const void *gate, const int32_t *q_var, const int32_t *kv_var, int topk, void *out,
                             float *lse, void *device_buf, size_t device_bytes, vsa_stream_t stream);

/* Failures inside the two host-buffer steps: the kernels of each head slice
 * record a timed-out internal wait in the status word of their staging
 * slot's workspace (as vsa_device_status describes for a caller's
 * workspace). This call synchronises `stream`, reads and clears both
 * slots' words in device_buf (desc, groups, topk and with_gate as in the
 * step's call) and sets *code to the first nonzero one (0 = no failure);
 * it returns VSA_ERR_DEVICE when *code != 0. The words are only ever set,
 * from 0, by a failing wait, so device_buf must be zeroed once before its
 * first use. */
vsa_status vsa_step_host_status(const vsa_desc *desc, int groups, int topk, int with_gate, void *device_buf,
                                vsa_stream_t stream, int32_t *code);

/* Human-readable name of a status. */
const char *vsa_status_string(vsa_status status);

/* Validation of the device-resident arguments, for debugging and for
 * callers that build their own indices: opt-in, never run by the other
 * calls (it synchronises `stream`). Checks, reading only inside the sizes
 * the descriptor and idx_cap declare:
 *   tile fills q_var / kv_var within [0, tile] (padded layouts; the key of
 *     KV tile j is valid iff its slot < kv_var[j], [FA4-adapt]
 *     _vbs_mask_mod), or, in TND, cu_seqlens_* non-negative, ascending,
 *     at most the total tokens, and no sequence longer than nQ (nKV)
 *     tiles ([NPU-test] actual_seq_lengths);
 *   if q_idx / q_cnt are given: every count within [0, idx_cap], the first
 *     count's entries within [0, nKV), ascending, each a tile with valid
 *     tokens ([FA4-adapt] _map_to_index and the vbs > 0 split of
 *     _build_sparse_tensors);
 *   if kv_ptr / kv_qidx are given: offsets start at 0, ascend and stay
 *     within nQ*idx_cap; entries within [0, nQ), ascending per KV tile; and
 *     with q_idx given too, the KV-owned index is exactly the transpose of
 *     the Q-owned one ([FA4-adapt] _build_sparse_tensors, KV-owned
 *     backward metadata).
 * q_var / kv_var are required in the padded layouts; each index is passed
 * whole or not at all (both pointers NULL). workspace: 256-byte aligned,
 * at least 256 bytes; only its status word is used. The first failing
 * check records its code (0xC001 bad q_var, 0xC002 bad kv_var, 0xC003 /
 * 0xC004 bad cu_seqlens_q / _kv, 0xC005 bad q_cnt, 0xC006 bad q_idx,
 * 0xC007 bad kv_ptr, 0xC008 bad kv_qidx, 0xC009 not a transpose) in the
 * status word; the call then reads and clears the word as
 * vsa_device_status does, sets *code and returns VSA_ERR_SHAPE for one of
 * these codes, VSA_ERR_DEVICE when the word already held another failure,
 * VSA_OK (code 0) when everything is in range. Host-side errors as for
 * vsa_build_block_map, VSA_ERR_WORKSPACE for the workspace, VSA_ERR_NULL
 * for code == NULL or half an index. */
vsa_status vsa_check_inputs(const vsa_desc *desc, const int32_t *q_var, const int32_t *kv_var,
                            const int32_t *q_idx, const int32_t *q_cnt, int idx_cap, const int32_t *kv_ptr,
                            const int32_t *kv_qidx, void *workspace, size_t workspace_bytes, vsa_stream_t stream,
                            int32_t *code);

/* Message of the last CUDA error behind a VSA_ERR_CUDA return, with the
 * name of the last kernel the library launched ("no error" if there was
 * none). The string is owned by the library (per calling thread). */
const char *vsa_last_cuda_error(void);

/* Synchronises `stream`, reads the device status word in `workspace` into
 * *code (0 = no failure; otherwise the site of the wait that timed out) and
 * clears it. Returns VSA_ERR_DEVICE when *code != 0. */
vsa_status vsa_device_status(void *workspace, vsa_stream_t stream, int32_t *code);

/* Instrumentation. While enabled, every kernel the library launches is
 * bracketed by CUDA events on its stream; vsa_profile_count / _name / _ms
 * read the records (synchronising on the events) and vsa_profile_reset
 * clears them. vsa_launch_count returns the number of kernels launched
 * since the library was loaded. */
void vsa_profile_enable(int on);
int vsa_profile_count(void);
const char *vsa_profile_name(int i);
float vsa_profile_ms(int i);
void vsa_profile_reset(void);
long long vsa_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* VSA_H */
