// paged_attention_decode_noalloc: the decode entry point for callers that
// cannot allocate device memory.
//
// Some callers of this library have no way to allocate: a serving engine that
// reserves the whole device up front for its KV pool and forbids allocation
// inside the decode loop, or a plug-in running inside a host framework that
// owns the device allocator and hands the plug-in only its input and output
// buffers.  Such a caller cannot provide the scratch workspace that
// paged_attention_decode asks for.  This variant uses a fixed scratch array
// compiled into the library instead.
//
// The scratch is a file-scope __device__ array, so every GPU that loads the
// library holds it (kScratchBytes) until the process exits.  Host code cannot
// use the array's name as a device address (in host code it is a host-side
// stand-in), so the device address is fetched with cudaGetSymbolAddress once
// per device, with that device current, on the first call made on it, and
// cached.  That first call on a device should come before any stream capture.
//
// The kernels keep no state in the scratch between calls: each call tags its
// piece counters with a fresh random 64-bit value (a counter of another tag
// counts as zero), and every partial result is written before it is read,
// so what an earlier call of another shape left there does not matter.  All calls share the one
// array, so calls whose work overlaps on the GPU (two streams, or two host
// threads) race on it and must be serialised by the caller.  The calling
// thread's current device must be the pool's (KV_EINVAL otherwise).
//
// This file calls no cudaMalloc, cudaFree or allocating library routine.
#include <mutex>

#include "pagedkv_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on device `dev`, which must be the
// current device (set up once per device).
cudaError_t scratch_for_device(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kv_status paged_attention_decode_noalloc(kv_pool_t pool, const void* q, void* out,
                                                    const int32_t* block_tables,
                                                    int max_blocks_per_seq, const int32_t* seq_lens,
                                                    int batch, int num_q_heads, float scale,
                                                    int num_kv_heads, void* stream) {
    const pagedkv::NvtxRange range("paged_attention_decode_noalloc");
    if (!pool) return KV_EINVAL;
    // the scratch, like the pool's tensor maps, must be the pool's device's
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_decode_noalloc");
    if (dev != pool->device) return KV_EINVAL;
    size_t need = 0;
    kv_status st = paged_attention_workspace_size(pool, batch, num_q_heads, &need);
    if (st != KV_OK) return st;
    if (need > kScratchBytes) return KV_ENOWORKSPACE;     // beyond the static maximum
    void* scratch = nullptr;
    e = scratch_for_device(dev, &scratch);
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_decode_noalloc(scratch)");
    return pagedkv::decode_with_workspace(pool, q, out, block_tables, max_blocks_per_seq, seq_lens,
                                          batch, num_q_heads, scale, num_kv_heads, scratch,
                                          kScratchBytes, static_cast<cudaStream_t>(stream));
}
