// host_step.cu -- one training step of the attention (block map, forward,
// backward) from host buffers, with the host<->device copies overlapped
// with the kernels.
//
// Pages: every head is an independent problem (Ascend
// test_npu_block_sparse_attention_backward.py, the per-(batch, head) loops of
// the TND/GQA golden; FastVideo test_vsa256_backward.py runs the step on
// [B, S, H, D] tensors). So the heads are cut into slices of whole GQA
// groups, each slice is copied into a compact device staging slot, and
// while slice g computes, slice g+1 streams in and slice g-1 streams out:
//
//   in-stream:      H2D(0)  H2D(1)  H2D(2) ...
//   caller stream:          step(0) step(1) step(2) ...
//   out-stream:                     D2H(0)  D2H(1) ...
//
// Every slice holds Hkv / groups key/value heads and their query heads.
// Nothing overlaps the first slice's copy in or the last slice's copy out,
// but slices of fewer heads do not shorten them: a BSHD head slice is a 2D
// copy of runs of heads*D*2 bytes, and the copy engines move 256-byte runs
// (one head) at about a third of the link's rate, 1,280-byte runs at ~80%.
//
// vsa_fwd_step_host is the same pipeline for inference (block map without
// the KV-owned index, forward; O and LSE come back).
// Two staging slots alternate; a slot's inputs are refilled once the step
// that read them is done, and its outputs are rewritten once their copy
// back is done (events). Within a slice the forward starts once q, k, v
// have landed (dO follows during it), O goes back during the backward and
// dk, dv during the dQ pass. A head slice is a strided 2D region of every
// layout (BSHD/TND: a run of Hs*D elements per token; BHSD: a run of
// Hs*S*D per batch entry), copied with cudaMemcpy2DAsync. The step per
// slice calls the same entry points as a device caller (vsa_build_block_map,
// vsa_fwd_reuse, and vsa_bwd_reuse through an internal variant that also
// marks when dk and dv are final, on the slice's descriptor), so results are
// bit-identical to running the whole problem on the device; with a gate, the
// gated compression branch runs too (its tile means are per head as well,
// and the three calls of a slice share its staging workspace, so q's and
// k's means are pooled once, by the block map, and v's once, by the
// forward). No
// device memory is allocated here: the caller provides the staging buffer.
#include <cstdint>

#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

struct SlotLayout {
    size_t ws, q, k, v, dO, out, dq, dk, dv, lse, map, qidx, qcnt, kvptr, kvqidx, ws_bytes, bytes;
    size_t gate, osp;  // gated compression branch only
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Sizes of one head slice (descriptor `s`: Hq and Hkv already divided).
SlotLayout slot_layout(const vsa_desc &s, int cap, bool gated) {
    SlotLayout L{};
    const size_t es = 2;
    const bool tnd = s.layout == VSA_LAYOUT_TND;
    const size_t tq = tnd ? (size_t)s.Sq : (size_t)s.B * s.Sq, tk = tnd ? (size_t)s.Skv : (size_t)s.B * s.Skv;
    const size_t qb = tq * s.Hq * s.D * es, kb = tk * s.Hkv * s.D * es;
    const size_t rows = (size_t)s.B * s.Hq * s.nQ;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    // the workspace first: its status word sits at the slot's start for
    // slices of every size
    L.ws_bytes = vsa_workspace_size(&s, gated ? 1 : 0);
    L.ws = take(L.ws_bytes);
    L.q = take(qb);
    L.k = take(kb);
    L.v = take(kb);
    L.dO = take(qb);
    L.out = take(qb);
    L.dq = take(qb);
    L.dk = take(kb);
    L.dv = take(kb);
    L.lse = take(tq * s.Hq * 4);
    L.map = take(rows * s.nKV);
    L.qidx = take(rows * cap * 4);
    L.qcnt = take(rows * 4);
    L.kvptr = take((size_t)s.B * s.Hq * (s.nKV + 1) * 4);
    L.kvqidx = take(rows * cap * 4);
    if (gated) {
        L.gate = take(qb);
        L.osp = take(qb);
    }
    L.bytes = off;
    return L;
}


// The slice of heads [h0, h0 + hs) of a [.., H, ..] tensor as a 2D copy:
// `rows` runs of `width` bytes, `pitch` bytes apart in the full tensor,
// starting `first` bytes in.
struct Strided {
    size_t rows, width, pitch, first;
};
Strided head_slice(const vsa_desc &d, bool q_side, int h0, int hs, size_t elem_bytes_per_token_head) {
    const int H = q_side ? d.Hq : d.Hkv;
    const int S = q_side ? d.Sq : d.Skv;
    const size_t e = elem_bytes_per_token_head;
    if (d.layout == VSA_LAYOUT_BHSD) return {(size_t)d.B, (size_t)hs * S * e, (size_t)H * S * e, (size_t)h0 * S * e};
    const size_t tokens = d.layout == VSA_LAYOUT_TND ? (size_t)S : (size_t)d.B * S;
    return {tokens, (size_t)hs * e, (size_t)H * e, (size_t)h0 * e};
}
// LSE [B, Hq, Sq] (TND: [Hq, T_q]) head slice.
Strided lse_slice(const vsa_desc &d, int h0, int hs) {
    if (d.layout == VSA_LAYOUT_TND) return {1, (size_t)hs * d.Sq * 4, (size_t)d.Hq * d.Sq * 4, (size_t)h0 * d.Sq * 4};
    return {(size_t)d.B, (size_t)hs * d.Sq * 4, (size_t)d.Hq * d.Sq * 4, (size_t)h0 * d.Sq * 4};
}

cudaError_t copy_in(void *dst, const void *host, const Strided &r, cudaStream_t s) {
    return cudaMemcpy2DAsync(dst, r.width, static_cast<const uint8_t *>(host) + r.first, r.pitch, r.width, r.rows,
                             cudaMemcpyHostToDevice, s);
}
cudaError_t copy_out(void *host, const void *src, const Strided &r, cudaStream_t s) {
    return cudaMemcpy2DAsync(static_cast<uint8_t *>(host) + r.first, r.pitch, src, r.width, r.width, r.rows,
                             cudaMemcpyDeviceToHost, s);
}

vsa_status check_groups(const vsa_desc *d, int groups, int topk, vsa_desc *slice, int *cap) {
    int q0 = 0, kv0 = 0;
    const vsa_status st = vsa_head_slice(d, groups, 0, slice, &q0, &kv0);
    if (st != VSA_OK) return st;
    if (topk < 1) return VSA_ERR_SHAPE;
    *cap = topk < d->nKV ? topk : d->nKV;
    return VSA_OK;
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" vsa_status vsa_head_slice(const vsa_desc *desc, int groups, int g, vsa_desc *slice, int32_t *q_head0,
                                     int32_t *kv_head0) {
    if (!desc || !slice || !q_head0 || !kv_head0) return VSA_ERR_NULL;
    Prob p;
    const vsa_status st = to_prob(desc, &p);  // every descriptor check of the other calls
    if (st != VSA_OK) return st;
    if (groups < 1 || desc->Hkv % groups != 0 || g < 0 || g >= groups) return VSA_ERR_SHAPE;
    *slice = *desc;
    slice->Hq = desc->Hq / groups;
    slice->Hkv = desc->Hkv / groups;
    *q_head0 = g * slice->Hq;
    *kv_head0 = g * slice->Hkv;
    return VSA_OK;
}

extern "C" size_t vsa_train_step_host_size(const vsa_desc *desc, int groups, int topk, int with_gate) {
    vsa_desc s;
    int cap = 0;
    if (check_groups(desc, groups, topk, &s, &cap) != VSA_OK) return 0;
    return 2 * slot_layout(s, cap, with_gate != 0).bytes;
}

namespace vsa {
namespace {

// The pipelined step; train == false runs the block map and the forward
// only (no dO in, no gradients out, no KV-owned index).
vsa_status step_host(const vsa_desc *desc, int groups, bool train, const void *q, const void *k, const void *v,
                     const void *dO, const void *gate, const int32_t *q_var, const int32_t *kv_var, int topk,
                     void *out, float *lse, void *dq, void *dk, void *dv, void *device_buf, size_t device_bytes,
                     vsa_stream_t stream) {
    vsa_desc sd;
    int cap = 0;
    const vsa_status st = check_groups(desc, groups, topk, &sd, &cap);
    if (st != VSA_OK) return st;
    if (!q || !k || !v) return VSA_ERR_NULL;
    if (train ? (!dO || !dq || !dk || !dv) : !out) return VSA_ERR_NULL;
    const bool gated = gate != nullptr;
    const SlotLayout L = slot_layout(sd, cap, gated);
    if (!device_buf || (reinterpret_cast<uintptr_t>(device_buf) & 255u) != 0 || device_bytes < 2 * L.bytes)
        return VSA_ERR_WORKSPACE;

    cudaStream_t sc = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t s_in = nullptr, s_out = nullptr;
    // per slot: q/k/v landed, dO landed, forward done, dk/dv final, step done, copies back done
    cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_in[2] = {}, ev_do[2] = {}, ev_fwd[2] = {}, ev_dkv[2] = {},
                ev_comp[2] = {}, ev_out[2] = {};
    vsa_status rc = VSA_OK;
    auto cu = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == VSA_OK) rc = status_from_cuda(e);
        return rc == VSA_OK;
    };
    auto vs = [&](vsa_status e) {
        if (e != VSA_OK && rc == VSA_OK) rc = e;
        return rc == VSA_OK;
    };
    const unsigned evf = cudaEventDisableTiming;
    bool ok = cu(cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking)) &&
              cu(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking)) &&
              cu(cudaEventCreateWithFlags(&ev_start, evf)) && cu(cudaEventCreateWithFlags(&ev_end, evf));
    for (int i = 0; ok && i < 2; ++i)
        ok = cu(cudaEventCreateWithFlags(&ev_in[i], evf)) && cu(cudaEventCreateWithFlags(&ev_do[i], evf)) &&
             cu(cudaEventCreateWithFlags(&ev_fwd[i], evf)) && cu(cudaEventCreateWithFlags(&ev_dkv[i], evf)) &&
             cu(cudaEventCreateWithFlags(&ev_comp[i], evf)) && cu(cudaEventCreateWithFlags(&ev_out[i], evf));
    // both side streams start after what the caller queued before this call
    ok = ok && cu(cudaEventRecord(ev_start, sc)) && cu(cudaStreamWaitEvent(s_in, ev_start, 0)) &&
         cu(cudaStreamWaitEvent(s_out, ev_start, 0));

    const size_t row = (size_t)desc->D * 2;  // bytes per (token, head)
    const vsa_desc &sg = sd;                 // every slice's problem
    const SlotLayout &Lg = L;
    for (int g = 0; ok && g < groups; ++g) {
        const int slot = g & 1, hq0 = g * sg.Hq, hk0 = g * sg.Hkv;  // the slice's first heads
        uint8_t *base = static_cast<uint8_t *>(device_buf) + slot * L.bytes;
        const Strided rq = head_slice(*desc, true, hq0, sg.Hq, row), rk = head_slice(*desc, false, hk0, sg.Hkv, row);
        // inputs of slice g; the slot's previous inputs were read by step g-2
        if (g >= 2) ok = cu(cudaStreamWaitEvent(s_in, ev_comp[slot], 0));
        // (q, k, v first: the block map and the forward start before dO lands)
        ok = ok && cu(copy_in(base + Lg.q, q, rq, s_in)) && cu(copy_in(base + Lg.k, k, rk, s_in)) &&
             cu(copy_in(base + Lg.v, v, rk, s_in));
        if (ok && gated) ok = cu(copy_in(base + Lg.gate, gate, rq, s_in));
        ok = ok && cu(cudaEventRecord(ev_in[slot], s_in));
        if (ok && train) ok = cu(copy_in(base + Lg.dO, dO, rq, s_in)) && cu(cudaEventRecord(ev_do[slot], s_in));
        // step g on the caller's stream; the slot's previous outputs were copied back
        ok = ok && cu(cudaStreamWaitEvent(sc, ev_in[slot], 0));
        if (ok && g >= 2) ok = cu(cudaStreamWaitEvent(sc, ev_out[slot], 0));
        if (!ok) break;
        uint8_t *ws = base + Lg.ws;
        int32_t *qidx = reinterpret_cast<int32_t *>(base + Lg.qidx), *qcnt = reinterpret_cast<int32_t *>(base + Lg.qcnt);
        int32_t *kvptr = reinterpret_cast<int32_t *>(base + Lg.kvptr);
        int32_t *kvqidx = reinterpret_cast<int32_t *>(base + Lg.kvqidx);
        float *lse_d = reinterpret_cast<float *>(base + Lg.lse);
        // gated: O (the sparse attention output) stays in its own buffer, out = O + gate (*) c
        const void *g_d = gated ? base + Lg.gate : nullptr;
        void *osp_d = gated ? base + Lg.osp : nullptr;
        ok = vs(vsa_build_block_map(&sg, base + Lg.q, base + Lg.k, q_var, kv_var, topk, train ? 1 : 0,
                                    base + Lg.map, qidx, qcnt, cap, train ? kvptr : nullptr, train ? kvqidx : nullptr,
                                    ws, Lg.ws_bytes, stream)) &&
             vs(vsa_fwd_reuse(&sg, base + Lg.q, base + Lg.k, base + Lg.v, qidx, qcnt, cap, q_var, kv_var, g_d,
                              base + Lg.out, lse_d, osp_d, VSA_REUSE_QK_MEANS, ws, Lg.ws_bytes, stream)) &&
             cu(cudaEventRecord(ev_fwd[slot], sc));
        if (ok && train)
            ok = cu(cudaStreamWaitEvent(sc, ev_do[slot], 0)) &&
                 vs(bwd_reuse_event(&sg, base + Lg.dO, base + Lg.q, base + Lg.k, base + Lg.v,
                                    gated ? osp_d : base + Lg.out, lse_d, qidx, qcnt, cap, kvptr, kvqidx, q_var,
                                    kv_var, g_d, base + Lg.dq, base + Lg.dk, base + Lg.dv,
                                    VSA_REUSE_QK_MEANS | VSA_REUSE_V_MEANS, ws, Lg.ws_bytes, stream, ev_dkv[slot]));
        ok = ok && cu(cudaEventRecord(ev_comp[slot], sc));
        // outputs of slice g: O and LSE are final after the forward, dk and
        // dv after the dK/dV pass (they go back while dQ is computed), dq at
        // the end of the step
        ok = ok && cu(cudaStreamWaitEvent(s_out, ev_fwd[slot], 0));
        if (ok && out) ok = cu(copy_out(out, base + Lg.out, rq, s_out));
        if (ok && lse) ok = cu(copy_out(lse, lse_d, lse_slice(*desc, hq0, sg.Hq), s_out));
        if (ok && train)
            ok = cu(cudaStreamWaitEvent(s_out, ev_dkv[slot], 0)) && cu(copy_out(dk, base + Lg.dk, rk, s_out)) &&
                 cu(copy_out(dv, base + Lg.dv, rk, s_out)) && cu(cudaStreamWaitEvent(s_out, ev_comp[slot], 0)) &&
                 cu(copy_out(dq, base + Lg.dq, rq, s_out));
        ok = ok && cu(cudaEventRecord(ev_out[slot], s_out));
    }
    // the caller's stream completes after the last copy back (and after the
    // input stream, so no copy outlives the call's work on its stream)
    if (s_in && s_out) {
        if (cudaEventRecord(ev_end, s_out) == cudaSuccess) cudaStreamWaitEvent(sc, ev_end, 0);
        if (cudaEventRecord(ev_start, s_in) == cudaSuccess) cudaStreamWaitEvent(sc, ev_start, 0);
    }
    // destruction is deferred by the runtime until the queued work is done
    for (int i = 0; i < 2; ++i) {
        if (ev_in[i]) cudaEventDestroy(ev_in[i]);
        if (ev_do[i]) cudaEventDestroy(ev_do[i]);
        if (ev_fwd[i]) cudaEventDestroy(ev_fwd[i]);
        if (ev_dkv[i]) cudaEventDestroy(ev_dkv[i]);
        if (ev_comp[i]) cudaEventDestroy(ev_comp[i]);
        if (ev_out[i]) cudaEventDestroy(ev_out[i]);
    }
    if (ev_start) cudaEventDestroy(ev_start);
    if (ev_end) cudaEventDestroy(ev_end);
    if (s_in) cudaStreamDestroy(s_in);
    if (s_out) cudaStreamDestroy(s_out);
    return rc;
}

}  // namespace
}  // namespace vsa

extern "C" vsa_status vsa_train_step_host(const vsa_desc *desc, int groups, const void *q, const void *k,
                                          const void *v, const void *dO, const void *gate, const int32_t *q_var,
                                          const int32_t *kv_var, int topk, void *out, float *lse, void *dq,
                                          void *dk, void *dv, void *device_buf, size_t device_bytes,
                                          vsa_stream_t stream) {
    return step_host(desc, groups, true, q, k, v, dO, gate, q_var, kv_var, topk, out, lse, dq, dk, dv, device_buf,
                     device_bytes, stream);
}

extern "C" vsa_status vsa_fwd_step_host(const vsa_desc *desc, int groups, const void *q, const void *k,
                                        const void *v, const void *gate, const int32_t *q_var, const int32_t *kv_var,
                                        int topk, void *out, float *lse, void *device_buf, size_t device_bytes,
                                        vsa_stream_t stream) {
    return step_host(desc, groups, false, q, k, v, nullptr, gate, q_var, kv_var, topk, out, lse, nullptr, nullptr,
                     nullptr, device_buf, device_bytes, stream);
}

extern "C" vsa_status vsa_step_host_status(const vsa_desc *desc, int groups, int topk, int with_gate,
                                           void *device_buf, vsa_stream_t stream, int32_t *code) {
    if (!device_buf || !code) return VSA_ERR_NULL;
    vsa_desc sd;
    int cap = 0;
    const vsa_status st = check_groups(desc, groups, topk, &sd, &cap);
    if (st != VSA_OK) return st;
    const SlotLayout L = slot_layout(sd, cap, with_gate != 0);
    *code = 0;
    for (int slot = 0; slot < 2; ++slot) {
        int32_t c = 0;
        const vsa_status r =
            vsa_device_status(static_cast<uint8_t *>(device_buf) + slot * L.bytes + L.ws, stream, &c);
        if (r != VSA_OK && r != VSA_ERR_DEVICE) return r;
        if (c != 0 && *code == 0) *code = c;
    }
    return *code ? VSA_ERR_DEVICE : VSA_OK;
}
