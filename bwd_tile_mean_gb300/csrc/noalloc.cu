// noalloc.cu -- vsa_build_block_map_static: the block-map step with its
// scratch (the fp32 tile means of q and k) held in a fixed device array
// that lives in this library, for callers that cannot allocate device
// memory (see include/vsa.h).
#include <mutex>

#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

// Scratch for the pooled tile means: B*Hq*nQ*D + B*Hkv*nKV*D floats at most.
constexpr size_t kStaticScratchFloats = size_t(4) << 20;  // 4 Mi floats = 16 MiB
__device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
float *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. Host code
// cannot use the array's name as a device pointer, so the address is looked
// up once per device with that device current and cached.
cudaError_t scratch_for_current_device(float **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<float *>(ptr);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" vsa_status vsa_build_block_map_static(const vsa_desc *desc, const void *q, const void *k,
                                                 const int32_t *q_var, const int32_t *kv_var, int topk,
                                                 int need_bwd_index, uint8_t *block_map, int32_t *q_idx,
                                                 int32_t *q_cnt, int idx_cap, int32_t *kv_ptr, int32_t *kv_qidx,
                                                 vsa_stream_t stream) {
    // Same host checks as vsa_build_block_map, minus the workspace.
    if (!desc) return VSA_ERR_NULL;
    if (desc->layout < 0 || desc->layout > 2) return VSA_ERR_LAYOUT;
    if (desc->dtype != VSA_DTYPE_BF16 && desc->dtype != VSA_DTYPE_FP16) return VSA_ERR_DTYPE;
    if (desc->B < 1 || desc->Hq < 1 || desc->Hkv < 1 || desc->Hq % desc->Hkv != 0) return VSA_ERR_SHAPE;
    if (desc->D != 128) return VSA_ERR_UNSUPPORTED;
    if ((desc->tile_q != 128 && desc->tile_q != 256) || (desc->tile_kv != 128 && desc->tile_kv != 256))
        return VSA_ERR_UNSUPPORTED;
    if (desc->nQ < 1 || desc->nKV < 1) return VSA_ERR_SHAPE;
    if (desc->layout == VSA_LAYOUT_TND) {
        if (!desc->cu_seqlens_q || !desc->cu_seqlens_kv) return VSA_ERR_MISSING_SEQLENS;
    } else {
        if ((long long)desc->Sq != (long long)desc->nQ * desc->tile_q ||
            (long long)desc->Skv != (long long)desc->nKV * desc->tile_kv)
            return VSA_ERR_SHAPE;
        if (!q_var || !kv_var) return VSA_ERR_NULL;
    }
    if (!q || !k || !block_map || !q_idx || !q_cnt) return VSA_ERR_NULL;
    if (need_bwd_index && (!kv_ptr || !kv_qidx)) return VSA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(k) & 15u)) return VSA_ERR_LAYOUT;
    if (topk < 1 || idx_cap < (topk < desc->nKV ? topk : desc->nKV)) return VSA_ERR_SHAPE;
    if (desc->nKV > kMaxSelectKV) return VSA_ERR_UNSUPPORTED;
    if (!(desc->scale >= 0.f)) return VSA_ERR_SHAPE;
    const size_t nq = (size_t)desc->B * desc->Hq * desc->nQ * desc->D;
    const size_t nk = (size_t)desc->B * desc->Hkv * desc->nKV * desc->D;
    if (nq + nk > kStaticScratchFloats) return VSA_ERR_SCRATCH;  // beyond the fixed scratch

    Prob p{};
    p.layout = desc->layout;
    p.dtype = desc->dtype;
    p.B = desc->B;
    p.Hq = desc->Hq;
    p.Hkv = desc->Hkv;
    p.D = desc->D;
    p.Sq = desc->Sq;
    p.Skv = desc->Skv;
    p.tile_q = desc->tile_q;
    p.tile_kv = desc->tile_kv;
    p.nQ = desc->nQ;
    p.nKV = desc->nKV;
    p.cu_q = desc->cu_seqlens_q;
    p.cu_kv = desc->cu_seqlens_kv;
    p.q_var = desc->layout == VSA_LAYOUT_TND ? nullptr : q_var;
    p.kv_var = desc->layout == VSA_LAYOUT_TND ? nullptr : kv_var;
    p.scale = desc->scale;

    float *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return VSA_ERR_CUDA;
    float *pq = scratch;
    float *pk = scratch + ((nq + 63) & ~size_t(63));
    if ((size_t)(pk - scratch) + nk > kStaticScratchFloats) return VSA_ERR_SCRATCH;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Every element of pq and pk is written by the pooling kernels before
    // it is read, so the array needs no clearing between calls.
    if (launch_pool_qkv(p, q, pq, k, pk, nullptr, nullptr, s) != cudaSuccess) return VSA_ERR_CUDA;
    if (launch_select(p, pq, pk, topk, block_map, q_idx, q_cnt, idx_cap, s) != cudaSuccess) return VSA_ERR_CUDA;
    if (need_bwd_index && launch_transpose(p, block_map, kv_ptr, kv_qidx, idx_cap, s) != cudaSuccess)
        return VSA_ERR_CUDA;
    return VSA_OK;
}
