// vsa_api.cu -- the C ABI of libvsa.so (include/vsa.h): host-side argument
// validation, workspace layout, tensor-map encoding, launch sequencing and
// instrumentation. No device memory is allocated here and nothing
// synchronises except vsa_device_status and the profile readers.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <utility>
#include <vector>

#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {

// --------------------------------------------------------- instrumentation
namespace {
struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
};
bool g_prof = false;
std::vector<ProfRec> g_recs;
std::vector<cudaEvent_t> g_free;
long long g_launches = 0;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

const char *g_last_launch = "";

void prof_begin(const char *name, cudaStream_t s) {
    ++g_launches;
    g_last_launch = name;
    if (!g_prof) return;
    ProfRec r{name, take_event(), take_event()};
    cudaEventRecord(r.a, s);
    g_recs.push_back(r);
}
void prof_end(cudaStream_t s) {
    if (!g_prof || g_recs.empty()) return;
    cudaEventRecord(g_recs.back().b, s);
}

// ------------------------------------------------------------ tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}
}  // namespace

// 4D map (D, S, H, B) over a q- or kv-shaped 16-bit tensor; box = 64 dims x
// 128 tokens of one head, 128-byte swizzle (the operand layout the tcgen05
// descriptors expect). TND maps (D, T, H, 1).
bool make_tmap_rows(CUtensorMap *map, const Prob &p, bool q_side, const void *base, int H, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = 2, S = (cuuint64_t)(q_side ? p.Sq : p.Skv), D = (cuuint64_t)p.D;
    cuuint64_t dims[4] = {D, S, (cuuint64_t)H, (cuuint64_t)(p.layout == L_TND ? 1 : p.B)};
    cuuint64_t strides[3];
    if (p.layout == L_BHSD) {
        strides[0] = D * es;
        strides[1] = S * D * es;
        strides[2] = (cuuint64_t)H * S * D * es;
    } else {
        strides[0] = (cuuint64_t)H * D * es;
        strides[1] = D * es;
        strides[2] = S * H * D * es;
    }
    cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1}, estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, p.dtype == T_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------ contexts, attributes
namespace {
PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    }
    return fn;
}
PFN_cuCtxGetId_v12000 ctx_id_fn() {
    static PFN_cuCtxGetId_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
    }
    return fn;
}
struct AttrSet {
    unsigned long long ctx;  // context id
    const void *kernel;
    int bytes;               // the limit set there
};
std::mutex g_attr_mu;
std::vector<AttrSet> g_attr_done;
}  // namespace

unsigned long long current_context_id() {
    auto cur = ctx_current_fn();
    auto idf = ctx_id_fn();
    if (!cur || !idf) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (cur(&c) != CUDA_SUCCESS || !c) return 0;
    if (idf(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

cudaError_t ensure_smem_limit(const void *kernel, int bytes) {
    // one lock over the check and the set: a thread that needs less cannot
    // set its limit after another thread raised it
    std::lock_guard<std::mutex> lock(g_attr_mu);
    unsigned long long ctx = current_context_id();
    if (ctx)
        for (const auto &e : g_attr_done)
            if (e.ctx == ctx && e.kernel == kernel && e.bytes >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    ctx = current_context_id();  // the call above brings the context up if it was not yet
    if (ctx) {
        bool found = false;
        for (auto &x : g_attr_done)
            if (x.ctx == ctx && x.kernel == kernel) {
                x.bytes = bytes;  // only ever raised: a smaller request returned above
                found = true;
            }
        if (!found) g_attr_done.push_back({ctx, kernel, bytes});
    }
    return cudaSuccess;
}

// -------------------------------------------------------------- validation
bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

vsa_status to_prob(const vsa_desc *d, Prob *p) {
    if (!d) return VSA_ERR_NULL;
    if (d->layout < 0 || d->layout > 2) return VSA_ERR_LAYOUT;
    if (d->dtype != VSA_DTYPE_BF16 && d->dtype != VSA_DTYPE_FP16) return VSA_ERR_DTYPE;
    if (d->B < 1 || d->Hq < 1 || d->Hkv < 1 || d->Hq % d->Hkv != 0) return VSA_ERR_SHAPE;
    if (d->D != 128) return VSA_ERR_UNSUPPORTED;
    if ((d->tile_q != 128 && d->tile_q != 256) || (d->tile_kv != 128 && d->tile_kv != 256))
        return VSA_ERR_UNSUPPORTED;
    if (d->nQ < 1 || d->nKV < 1 || d->Sq < 0 || d->Skv < 0) return VSA_ERR_SHAPE;
    if (d->layout == VSA_LAYOUT_TND) {
        if (!d->cu_seqlens_q || !d->cu_seqlens_kv) return VSA_ERR_MISSING_SEQLENS;
    } else if ((long long)d->Sq != (long long)d->nQ * d->tile_q ||
               (long long)d->Skv != (long long)d->nKV * d->tile_kv) {
        return VSA_ERR_SHAPE;
    }
    if (!(d->scale >= 0.f) || std::isinf(d->scale)) return VSA_ERR_SHAPE;
    p->layout = d->layout;
    p->dtype = d->dtype;
    p->B = d->B;
    p->Hq = d->Hq;
    p->Hkv = d->Hkv;
    p->D = d->D;
    p->Sq = d->Sq;
    p->Skv = d->Skv;
    p->tile_q = d->tile_q;
    p->tile_kv = d->tile_kv;
    p->nQ = d->nQ;
    p->nKV = d->nKV;
    p->cu_q = d->cu_seqlens_q;
    p->cu_kv = d->cu_seqlens_kv;
    p->q_var = nullptr;
    p->kv_var = nullptr;
    p->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->D);
    return VSA_OK;
}

vsa_status need_vars(const Prob &p, const int32_t *q_var, const int32_t *kv_var, Prob *out, bool need_q) {
    *out = p;
    if (p.layout == L_TND) return VSA_OK;
    if ((need_q && !q_var) || !kv_var) return VSA_ERR_NULL;
    out->q_var = q_var;
    out->kv_var = kv_var;
    return VSA_OK;
}

vsa_status block_map_prob(const vsa_desc *desc, const void *q, const void *k, const int32_t *q_var,
                          const int32_t *kv_var, int topk, int need_bwd_index, const uint8_t *block_map,
                          const int32_t *q_idx, const int32_t *q_cnt, int idx_cap, const int32_t *kv_ptr,
                          const int32_t *kv_qidx, Prob *p) {
    Prob p0;
    vsa_status st = to_prob(desc, &p0);
    if (st != VSA_OK) return st;
    if ((st = need_vars(p0, q_var, kv_var, p, true)) != VSA_OK) return st;
    if (!q || !k || !block_map || !q_idx || !q_cnt) return VSA_ERR_NULL;
    if (need_bwd_index && (!kv_ptr || !kv_qidx)) return VSA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k)) return VSA_ERR_LAYOUT;
    if (topk < 1 || idx_cap < (topk < p->nKV ? topk : p->nKV)) return VSA_ERR_SHAPE;
    if (p->nKV > kMaxSelectKV) return VSA_ERR_UNSUPPORTED;
    return VSA_OK;
}

vsa_status run_block_map(const Prob &p, const void *q, const void *k, int topk, int need_bwd_index,
                         uint8_t *block_map, int32_t *q_idx, int32_t *q_cnt, int idx_cap, int32_t *kv_ptr,
                         int32_t *kv_qidx, float *pq, float *pk, cudaStream_t s) {
    cudaError_t e = launch_pool_qkv(p, q, pq, k, pk, nullptr, nullptr, s);
    if (e == cudaSuccess) e = launch_select(p, pq, pk, topk, block_map, q_idx, q_cnt, idx_cap, s);
    if (e == cudaSuccess && need_bwd_index) e = launch_transpose(p, block_map, kv_ptr, kv_qidx, idx_cap, s);
    return status_from_cuda(e);
}

namespace {

struct WsLayout {
    size_t pq, pk, pv, c, nlse2, ndvec, redo, order, okeys, dc, A, ds, dpq, dpk, dpv, total;
};

WsLayout ws_layout(const Prob &p, bool gate) {
    WsLayout L{};
    size_t off = 256;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    const size_t fq = (size_t)p.B * p.Hq * p.nQ * p.D * 4, fk = (size_t)p.B * p.Hkv * p.nKV * p.D * 4;
    const size_t slots = (size_t)p.B * p.Hq * p.nQ * p.tile_q;  // padded tile layout
    L.pq = take(fq);
    L.pk = take(fk);
    L.nlse2 = take(slots * 4);
    L.ndvec = take(slots * 4);
    L.redo = take((size_t)p.B * p.Hq * p.nQ);
    L.order = take((size_t)dk_units(p) * 4);
    L.okeys = take((size_t)dk_units(p) * 4);
    if (gate) {
        L.pv = take(fk);
        L.c = take(fq);
        L.dc = take(fq);
        L.A = take((size_t)p.B * p.Hq * p.nQ * p.nKV * 4);
        L.ds = take((size_t)p.B * p.Hq * p.nQ * p.nKV * 4);
        L.dpq = take(fq);
        L.dpk = take(fk);
        L.dpv = take(fk);
    }
    L.total = off;
    return L;
}

vsa_status check_ws(const Prob &p, bool gate, void *ws, size_t bytes) {
    if (!ws) return VSA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return VSA_ERR_WORKSPACE;
    if (bytes < ws_layout(p, gate).total) return VSA_ERR_WORKSPACE;
    return VSA_OK;
}

template <typename X>
X *at(void *ws, size_t off) {
    return reinterpret_cast<X *>(reinterpret_cast<uint8_t *>(ws) + off);
}

cudaError_t g_last_cuda = cudaSuccess;

vsa_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return VSA_OK;
    g_last_cuda = e;
    return VSA_ERR_CUDA;
}

#define VSA_TRY(expr)                              \
    do {                                           \
        vsa_status _st = (expr);                   \
        if (_st != VSA_OK) return _st;             \
    } while (0)
#define VSA_CUDA(expr) VSA_TRY(cuda_status(expr))

}  // namespace

vsa_status status_from_cuda(cudaError_t e) { return cuda_status(e); }

}  // namespace vsa

using namespace vsa;

extern "C" {

size_t vsa_workspace_size(const vsa_desc *desc, int with_gate) {
    Prob p;
    if (to_prob(desc, &p) != VSA_OK) return 0;
    return ws_layout(p, with_gate != 0).total;
}

vsa_status vsa_build_block_map(const vsa_desc *desc, const void *q, const void *k, const int32_t *q_var,
                               const int32_t *kv_var, int topk, int need_bwd_index, uint8_t *block_map,
                               int32_t *q_idx, int32_t *q_cnt, int idx_cap, int32_t *kv_ptr, int32_t *kv_qidx,
                               void *workspace, size_t workspace_bytes, vsa_stream_t stream) {
    Prob p;
    VSA_TRY(block_map_prob(desc, q, k, q_var, kv_var, topk, need_bwd_index, block_map, q_idx, q_cnt, idx_cap,
                           kv_ptr, kv_qidx, &p));
    VSA_TRY(check_ws(p, false, workspace, workspace_bytes));
    const WsLayout L = ws_layout(p, false);
    return run_block_map(p, q, k, topk, need_bwd_index, block_map, q_idx, q_cnt, idx_cap, kv_ptr, kv_qidx,
                         at<float>(workspace, L.pq), at<float>(workspace, L.pk),
                         reinterpret_cast<cudaStream_t>(stream));
}

vsa_status vsa_mask_to_index(const vsa_desc *desc, const uint8_t *block_map, const int32_t *q_var,
                             const int32_t *kv_var, int need_bwd_index, int32_t *q_idx, int32_t *q_cnt, int idx_cap,
                             int32_t *kv_ptr, int32_t *kv_qidx, vsa_stream_t stream) {
    Prob p0, p;
    VSA_TRY(to_prob(desc, &p0));
    VSA_TRY(need_vars(p0, q_var, kv_var, &p, false));
    if (!block_map || !q_idx || !q_cnt) return VSA_ERR_NULL;
    if (need_bwd_index && (!kv_ptr || !kv_qidx)) return VSA_ERR_NULL;
    if (idx_cap < p.nKV) return VSA_ERR_SHAPE;
    if (p.nKV > 16000) return VSA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    VSA_CUDA(launch_mask_index(p, block_map, q_idx, q_cnt, idx_cap, s));
    if (need_bwd_index) VSA_CUDA(launch_transpose(p, block_map, kv_ptr, kv_qidx, idx_cap, s));
    return VSA_OK;
}

namespace {
vsa_status fwd_impl(const vsa_desc *desc, const void *q, const void *k, const void *v, const int32_t *q_idx,
                    const int32_t *q_cnt, const int32_t *q_sub, int block_q, int idx_cap, const int32_t *q_var,
                    const int32_t *kv_var, const void *gate, void *out, float *lse, void *o_sparse, int reuse,
                    void *workspace, size_t workspace_bytes, vsa_stream_t stream) {
    if ((reuse & ~(VSA_REUSE_QK_MEANS | VSA_REUSE_V_MEANS)) != 0) return VSA_ERR_SHAPE;
    Prob p0, p;
    VSA_TRY(to_prob(desc, &p0));
    VSA_TRY(need_vars(p0, q_var, kv_var, &p, gate != nullptr));
    if (!q || !k || !v || !q_idx || !q_cnt || !out || !lse) return VSA_ERR_NULL;
    if (gate && (!o_sparse || o_sparse == out)) return VSA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (gate && !aligned16(gate)) ||
        (o_sparse && !aligned16(o_sparse)))
        return VSA_ERR_LAYOUT;
    if (idx_cap < 1 || idx_cap > p.nKV) return VSA_ERR_SHAPE;
    if ((long long)idx_cap * (p.tile_kv / 128) > kMaxChunks) return VSA_ERR_UNSUPPORTED;
    VSA_TRY(check_ws(p, gate != nullptr, workspace, workspace_bytes));
    const WsLayout L = ws_layout(p, gate != nullptr);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    FwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.q_idx = q_idx;
    a.q_cnt = q_cnt;
    a.cap = idx_cap;
    a.out = out;
    a.o_sparse = o_sparse ? o_sparse : out;
    a.lse = lse;
    a.gate = gate;
    a.q_sub = q_sub;
    a.block_q = block_q;
    a.err = at<unsigned>(workspace, 0);
    a.redo = at<uint8_t>(workspace, L.redo);
    if (gate) {
        float *pq = at<float>(workspace, L.pq), *pk = at<float>(workspace, L.pk), *pv = at<float>(workspace, L.pv);
        const bool qk = (reuse & VSA_REUSE_QK_MEANS) == 0, vv = (reuse & VSA_REUSE_V_MEANS) == 0;
        VSA_CUDA(launch_pool_qkv(p, qk ? q : nullptr, pq, qk ? k : nullptr, pk, vv ? v : nullptr, pv, s));
        a.c = at<float>(workspace, L.c);
        VSA_CUDA(launch_compress_fwd(p, pq, pk, pv, const_cast<float *>(a.c), s));
    }
    VSA_CUDA(launch_fwd(p, a, s));
    return VSA_OK;
}
}  // namespace

vsa_status vsa_fwd(const vsa_desc *desc, const void *q, const void *k, const void *v, const int32_t *q_idx,
                   const int32_t *q_cnt, int idx_cap, const int32_t *q_var, const int32_t *kv_var,
                   const void *gate, void *out, float *lse, void *o_sparse, void *workspace,
                   size_t workspace_bytes, vsa_stream_t stream) {
    return fwd_impl(desc, q, k, v, q_idx, q_cnt, nullptr, 0, idx_cap, q_var, kv_var, gate, out, lse, o_sparse, 0,
                    workspace, workspace_bytes, stream);
}

vsa_status vsa_fwd_reuse(const vsa_desc *desc, const void *q, const void *k, const void *v, const int32_t *q_idx,
                         const int32_t *q_cnt, int idx_cap, const int32_t *q_var, const int32_t *kv_var,
                         const void *gate, void *out, float *lse, void *o_sparse, int reuse, void *workspace,
                         size_t workspace_bytes, vsa_stream_t stream) {
    return fwd_impl(desc, q, k, v, q_idx, q_cnt, nullptr, 0, idx_cap, q_var, kv_var, gate, out, lse, o_sparse,
                    reuse, workspace, workspace_bytes, stream);
}

vsa_status vsa_fwd_blocks(const vsa_desc *desc, int block_q, const void *q, const void *k, const void *v,
                          const int32_t *q_idx, const int32_t *q_cnt, const int32_t *q_sub, int idx_cap,
                          const int32_t *q_var, const int32_t *kv_var, void *out, float *lse, void *workspace,
                          size_t workspace_bytes, vsa_stream_t stream) {
    if (!desc || !q_sub) return VSA_ERR_NULL;
    if (block_q < 32 || block_q > desc->tile_q || desc->tile_q % block_q != 0 || block_q % 32 != 0)
        return VSA_ERR_SHAPE;
    return fwd_impl(desc, q, k, v, q_idx, q_cnt, q_sub, block_q, idx_cap, q_var, kv_var, nullptr, out, lse,
                    nullptr, 0, workspace, workspace_bytes, stream);
}

vsa_status vsa_gate_grad(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                         const int32_t *q_var, const int32_t *kv_var, void *dgate, void *workspace,
                         size_t workspace_bytes, vsa_stream_t stream) {
    Prob p0, p;
    VSA_TRY(to_prob(desc, &p0));
    VSA_TRY(need_vars(p0, q_var, kv_var, &p, true));
    if (!dO || !q || !k || !v || !dgate) return VSA_ERR_NULL;
    if (!aligned16(dO) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dgate))
        return VSA_ERR_LAYOUT;
    VSA_TRY(check_ws(p, true, workspace, workspace_bytes));
    const WsLayout L = ws_layout(p, true);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float *pq = at<float>(workspace, L.pq), *pk = at<float>(workspace, L.pk), *pv = at<float>(workspace, L.pv);
    float *c = at<float>(workspace, L.c);
    VSA_CUDA(launch_pool_qkv(p, q, pq, k, pk, v, pv, s));
    VSA_CUDA(launch_compress_fwd(p, pq, pk, pv, c, s));
    VSA_CUDA(launch_gate_grad(p, dO, c, dgate, s));
    return VSA_OK;
}

namespace {
vsa_status bwd_impl(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                    const void *o_sparse, const float *lse, const int32_t *q_idx, const int32_t *q_cnt,
                    const int32_t *q_sub, int block_q, int idx_cap, const int32_t *kv_ptr, const int32_t *kv_qidx,
                    const int32_t *kv_qsub, const int32_t *q_var, const int32_t *kv_var, const void *gate,
                    void *dq, void *dk, void *dv, int reuse, void *workspace, size_t workspace_bytes,
                    vsa_stream_t stream, cudaEvent_t dkdv_done = nullptr) {
    if ((reuse & ~(VSA_REUSE_QK_MEANS | VSA_REUSE_V_MEANS)) != 0) return VSA_ERR_SHAPE;
    Prob p0, p;
    VSA_TRY(to_prob(desc, &p0));
    VSA_TRY(need_vars(p0, q_var, kv_var, &p, true));
    if (!dO || !q || !k || !v || !o_sparse || !lse || !q_idx || !q_cnt || !kv_ptr || !kv_qidx || !dq || !dk ||
        !dv)
        return VSA_ERR_NULL;
    if (!aligned16(dO) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_sparse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (gate && !aligned16(gate)))
        return VSA_ERR_LAYOUT;
    if (idx_cap < 1 || idx_cap > p.nKV) return VSA_ERR_SHAPE;
    if ((long long)idx_cap * (p.tile_kv / 128) > kMaxChunks) return VSA_ERR_UNSUPPORTED;
    VSA_TRY(check_ws(p, gate != nullptr, workspace, workspace_bytes));
    const WsLayout L = ws_layout(p, gate != nullptr);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    BwdArgs a{};
    a.dO = dO;
    a.q = q;
    a.k = k;
    a.v = v;
    a.q_idx = q_idx;
    a.q_cnt = q_cnt;
    a.cap = idx_cap;
    a.kv_ptr = kv_ptr;
    a.kv_qidx = kv_qidx;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.q_sub = q_sub;
    a.kv_qsub = kv_qsub;
    a.block_q = block_q;
    a.err = at<unsigned>(workspace, 0);
    float *ndvec = at<float>(workspace, L.ndvec), *nlse2 = at<float>(workspace, L.nlse2);
    a.ndvec = ndvec;
    a.nlse2 = nlse2;
    VSA_CUDA(launch_bwd_prep(p, dO, o_sparse, lse, nlse2, ndvec, a.err, s));
    if (gate) {
        float *pq = at<float>(workspace, L.pq), *pk = at<float>(workspace, L.pk), *pv = at<float>(workspace, L.pv);
        const bool qk = (reuse & VSA_REUSE_QK_MEANS) == 0, vv = (reuse & VSA_REUSE_V_MEANS) == 0;
        VSA_CUDA(launch_pool_qkv(p, qk ? q : nullptr, pq, qk ? k : nullptr, pk, vv ? v : nullptr, pv, s));
        float *dpq = at<float>(workspace, L.dpq), *dpk = at<float>(workspace, L.dpk),
              *dpv = at<float>(workspace, L.dpv);
        VSA_CUDA(launch_compress_bwd(p, dO, gate, pq, pk, pv, at<float>(workspace, L.dc), at<float>(workspace, L.A),
                                     at<float>(workspace, L.ds), dpq, dpk, dpv, s));
        a.dpq = dpq;
        a.dpk = dpk;
        a.dpv = dpv;
    }
    int *order = at<int>(workspace, L.order);
    VSA_CUDA(launch_dk_order(p, kv_ptr, idx_cap, order, at<int>(workspace, L.okeys), s));
    a.dk_order = order;
    VSA_CUDA(launch_bwd_dkdv(p, a, s));
    if (dkdv_done) VSA_CUDA(cudaEventRecord(dkdv_done, s));  // dk, dv final before dQ's pass
    VSA_CUDA(launch_bwd_dq(p, a, s));
    return VSA_OK;
}
}  // namespace

vsa_status vsa_bwd(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                   const void *o_sparse, const float *lse, const int32_t *q_idx, const int32_t *q_cnt, int idx_cap,
                   const int32_t *kv_ptr, const int32_t *kv_qidx, const int32_t *q_var, const int32_t *kv_var,
                   const void *gate, void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                   vsa_stream_t stream) {
    return bwd_impl(desc, dO, q, k, v, o_sparse, lse, q_idx, q_cnt, nullptr, 0, idx_cap, kv_ptr, kv_qidx, nullptr,
                    q_var, kv_var, gate, dq, dk, dv, 0, workspace, workspace_bytes, stream);
}

vsa_status vsa_bwd_reuse(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                         const void *o_sparse, const float *lse, const int32_t *q_idx, const int32_t *q_cnt,
                         int idx_cap, const int32_t *kv_ptr, const int32_t *kv_qidx, const int32_t *q_var,
                         const int32_t *kv_var, const void *gate, void *dq, void *dk, void *dv, int reuse,
                         void *workspace, size_t workspace_bytes, vsa_stream_t stream) {
    return bwd_impl(desc, dO, q, k, v, o_sparse, lse, q_idx, q_cnt, nullptr, 0, idx_cap, kv_ptr, kv_qidx, nullptr,
                    q_var, kv_var, gate, dq, dk, dv, reuse, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace vsa {
vsa_status bwd_reuse_event(const vsa_desc *desc, const void *dO, const void *q, const void *k, const void *v,
                           const void *o_sparse, const float *lse, const int32_t *q_idx, const int32_t *q_cnt,
                           int idx_cap, const int32_t *kv_ptr, const int32_t *kv_qidx, const int32_t *q_var,
                           const int32_t *kv_var, const void *gate, void *dq, void *dk, void *dv, int reuse,
                           void *workspace, size_t workspace_bytes, vsa_stream_t stream, cudaEvent_t dkdv_done) {
    return bwd_impl(desc, dO, q, k, v, o_sparse, lse, q_idx, q_cnt, nullptr, 0, idx_cap, kv_ptr, kv_qidx, nullptr,
                    q_var, kv_var, gate, dq, dk, dv, reuse, workspace, workspace_bytes, stream, dkdv_done);
}
}  // namespace vsa

extern "C" {

vsa_status vsa_bwd_blocks(const vsa_desc *desc, int block_q, const void *dO, const void *q, const void *k,
                          const void *v, const void *out, const float *lse, const int32_t *q_idx,
                          const int32_t *q_cnt, const int32_t *q_sub, int idx_cap, const int32_t *kv_ptr,
                          const int32_t *kv_qidx, const int32_t *kv_qsub, const int32_t *q_var,
                          const int32_t *kv_var, void *dq, void *dk, void *dv, void *workspace,
                          size_t workspace_bytes, vsa_stream_t stream) {
    if (!desc || !q_sub || !kv_qsub) return VSA_ERR_NULL;
    if (block_q < 32 || block_q > desc->tile_q || desc->tile_q % block_q != 0 || block_q % 32 != 0)
        return VSA_ERR_SHAPE;
    return bwd_impl(desc, dO, q, k, v, out, lse, q_idx, q_cnt, q_sub, block_q, idx_cap, kv_ptr, kv_qidx, kv_qsub,
                    q_var, kv_var, nullptr, dq, dk, dv, 0, workspace, workspace_bytes, stream);
}

vsa_status vsa_mask_to_index_blocks(const vsa_desc *desc, int block_q, int nQb, const uint8_t *block_mask,
                                    const int32_t *q_var, const int32_t *kv_var, int need_bwd_index,
                                    uint8_t *tile_map, int32_t *q_idx, int32_t *q_cnt, int32_t *q_sub, int idx_cap,
                                    int32_t *kv_ptr, int32_t *kv_qidx, int32_t *kv_qsub, vsa_stream_t stream) {
    Prob p0, p;
    VSA_TRY(to_prob(desc, &p0));
    VSA_TRY(need_vars(p0, q_var, kv_var, &p, false));
    if (!block_mask || !tile_map || !q_idx || !q_cnt || !q_sub) return VSA_ERR_NULL;
    if (need_bwd_index && (!kv_ptr || !kv_qidx || !kv_qsub)) return VSA_ERR_NULL;
    if (block_q < 32 || block_q > p.tile_q || p.tile_q % block_q != 0 || block_q % 32 != 0) return VSA_ERR_SHAPE;
    if (nQb < 1 || nQb > p.nQ * (p.tile_q / block_q)) return VSA_ERR_SHAPE;
    if (idx_cap < p.nKV) return VSA_ERR_SHAPE;
    if (p.nKV > 16000) return VSA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    VSA_CUDA(launch_block_index(p, block_q, nQb, block_mask, tile_map, q_idx, q_cnt, q_sub, idx_cap,
                                need_bwd_index ? kv_ptr : nullptr, kv_qidx, kv_qsub, s));
    return VSA_OK;
}

const char *vsa_status_string(vsa_status st) {
    switch (st) {
        case VSA_OK: return "ok";
        case VSA_ERR_NULL: return "a required pointer is NULL";
        case VSA_ERR_SHAPE: return "inconsistent sizes, or an index or tile fill out of range";
        case VSA_ERR_DTYPE: return "unsupported dtype (bf16 or fp16 only)";
        case VSA_ERR_LAYOUT: return "unknown layout or misaligned pointer";
        case VSA_ERR_UNSUPPORTED: return "unsupported size (D must be 128, tiles 128 or 256)";
        case VSA_ERR_MISSING_SEQLENS: return "TND layout needs cu_seqlens_q and cu_seqlens_kv";
        case VSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case VSA_ERR_CUDA: return "CUDA launch or runtime error";
        case VSA_ERR_DEVICE: return "a kernel reported a failed internal wait";
        case VSA_ERR_SCRATCH: return "problem exceeds the fixed scratch of vsa_build_block_map_static";
    }
    return "unknown status";
}

vsa_status vsa_device_status(void *workspace, vsa_stream_t stream, int32_t *code) {
    if (!workspace || !code) return VSA_ERR_NULL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VSA_ERR_CUDA;
    if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return VSA_ERR_CUDA;
    if (v != 0 && cudaMemset(workspace, 0, sizeof(v)) != cudaSuccess) return VSA_ERR_CUDA;
    *code = (int32_t)v;
    return v ? VSA_ERR_DEVICE : VSA_OK;
}

const char *vsa_last_cuda_error(void) {
    static thread_local char buf[256];
    if (g_last_cuda == cudaSuccess) return "no error";
    snprintf(buf, sizeof(buf), "%s (last kernel launched: %s)", cudaGetErrorString(g_last_cuda), g_last_launch);
    return buf;
}

void vsa_profile_enable(int on) { g_prof = on != 0; }
int vsa_profile_count(void) { return (int)g_recs.size(); }
const char *vsa_profile_name(int i) {
    return (i >= 0 && i < (int)g_recs.size()) ? g_recs[i].name : "";
}
float vsa_profile_ms(int i) {
    if (i < 0 || i >= (int)g_recs.size()) return -1.f;
    float ms = -1.f;
    cudaEventSynchronize(g_recs[i].b);
    cudaEventElapsedTime(&ms, g_recs[i].a, g_recs[i].b);
    return ms;
}
void vsa_profile_reset(void) {
    for (auto &r : g_recs) {
        g_free.push_back(r.a);
        g_free.push_back(r.b);
    }
    g_recs.clear();
}
long long vsa_launch_count(void) { return g_launches; }

}  // extern "C"
