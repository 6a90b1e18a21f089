// noalloc.cu -- vsa_build_block_map_static: the block-map step with its
// scratch (the fp32 tile means of q and k) held in a fixed device array
// that lives in this library, for callers that cannot allocate device
// memory (see include/vsa.h). Argument checks and launches are those of
// vsa_build_block_map; only where the tile means live differs.
#include <mutex>

#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

// Scratch for the pooled tile means: B*Hq*nQ*D + B*Hkv*nKV*D floats at most
// (plus at most 63 floats of alignment padding between the two).
constexpr size_t kStaticScratchFloats = size_t(4) << 20;  // 4 Mi floats = 16 MiB
__device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 128;
struct ScratchAddr {
    unsigned long long ctx;  // context the address belongs to (0: not looked up yet)
    float *ptr;
};
std::mutex g_mu;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array in the current device's context. In
// host code the array's name stands for a host-side shadow, not a device
// address, so the address is looked up (cudaGetSymbolAddress, with the
// device current) the first time a device is used and kept. The entry is
// keyed by the context's id: after a device reset the device runs a new
// context in which the module, and so the array, is loaded afresh, and the
// look-up is done again.
cudaError_t scratch_for_current_device(float **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchAddr &slot = g_scratch_addr[dev];
    const unsigned long long ctx = current_context_id();
    if (slot.ptr == nullptr || ctx == 0 || ctx != slot.ctx) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) return e;
        slot.ptr = static_cast<float *>(ptr);
        slot.ctx = current_context_id();  // the look-up brings the context up if it was not yet
    }
    *out = slot.ptr;
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
    Prob p;
    const vsa_status st = block_map_prob(desc, q, k, q_var, kv_var, topk, need_bwd_index, block_map, q_idx, q_cnt,
                                         idx_cap, kv_ptr, kv_qidx, &p);
    if (st != VSA_OK) return st;
    const size_t nq = (size_t)p.B * p.Hq * p.nQ * p.D;
    const size_t nk = (size_t)p.B * p.Hkv * p.nKV * p.D;
    const size_t pk_off = (nq + 63) & ~size_t(63);  // 256-byte aligned start of the key means
    if (pk_off + nk > kStaticScratchFloats) return VSA_ERR_SCRATCH;  // beyond the fixed scratch

    float *scratch = nullptr;
    const cudaError_t e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) return status_from_cuda(e);
    // Every element of the two mean arrays is written by the pooling kernel
    // before the selection reads it, so the array needs no clearing.
    return run_block_map(p, q, k, topk, need_bwd_index, block_map, q_idx, q_cnt, idx_cap, kv_ptr, kv_qidx, scratch,
                         scratch + pk_off, reinterpret_cast<cudaStream_t>(stream));
}
