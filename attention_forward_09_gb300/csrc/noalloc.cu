// noalloc.cu -- attn_fwd_paged_noalloc: paged decode without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// the decode: code being recorded into a CUDA graph (cudaMalloc is not
// allowed inside a stream capture), plugins hosted by a framework that owns
// all device memory and exposes no allocator to them, and servers that fix
// their memory budget at start-up and forbid any later allocation.  For
// them this entry point supplies the split-K scratch itself, from one
// file-scope device array, and otherwise runs exactly attn_fwd_paged.
//
// The array is device memory of every GPU on which this library's code is
// loaded, held until the process exits.  Its host-side name is only a
// stand-in: the device address is looked up with cudaGetSymbolAddress on
// the first call on each device (with that device current) and cached for
// the life of the process.  cudaDeviceReset unloads the library's device
// code, after which the array may live elsewhere: the cache does not notice,
// so the entry point must not be used on a device after it was reset.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gbattn.h"

namespace {

constexpr size_t kScratchBytes = GBATTN_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; keeps the previous call's contents.
static __device__ __align__(256) unsigned char g_paged_scratch[kScratchBytes];

// Device address of g_paged_scratch on the current device (set up once per device).
gbattn_status scratch_address(void** out) {
    static void* addr[64];
    static bool have[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GBATTN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return GBATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_paged_scratch) != cudaSuccess || p == nullptr) return GBATTN_ERR_CUDA;
        addr[dev] = p;
        have[dev] = true;
    }
    *out = addr[dev];
    return GBATTN_OK;
}

}  // namespace

extern "C" gbattn_status attn_fwd_paged_noalloc(const void* q, const void* kv_cache, int num_blocks, int block_size,
                                                const int32_t* block_table, int max_blocks_per_seq,
                                                const int32_t* seq_lens, int num_seqs, int max_seq_len, int Hq,
                                                int Hkv, int D, float softmax_scale, int causal, void* out,
                                                gbattn_dtype out_dtype, float* lse, uint32_t* dev_status,
                                                void* stream) {
    // Sizes whose scratch would not fit are refused before anything touches the GPU.
    if (attn_fwd_paged_workspace_size(num_seqs, Hq, Hkv, D, max_seq_len) > kScratchBytes)
        return GBATTN_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    const gbattn_status s = scratch_address(&scratch);
    if (s != GBATTN_OK) return s;
    // Nothing in the scratch has to start at zero: the schedule kernel resets
    // its work counter and every partial result is written before it is read.
    return attn_fwd_paged(q, kv_cache, num_blocks, block_size, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                          max_seq_len, Hq, Hkv, D, softmax_scale, causal, out, out_dtype, lse, scratch, kScratchBytes,
                          dev_status, stream);
}
