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
// The kernels keep no state in the scratch between calls: every call writes
// what it later reads, so nothing needs clearing.  All calls share the one
// array, so calls whose work overlaps on the GPU (two streams, or two host
// threads) race on it and must be serialised by the caller.
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

// Device address of g_decode_scratch on the current device (set up once).
cudaError_t scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
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
    size_t need = 0;
    kv_status st = paged_attention_workspace_size(pool, batch, num_q_heads, &need);
    if (st != KV_OK) return st;
    if (need > kScratchBytes) return KV_ENOWORKSPACE;     // beyond the static maximum
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return KV_ECUDA;
    return paged_attention_decode(pool, q, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                                  num_q_heads, scale, num_kv_heads, scratch, kScratchBytes, stream);
}
