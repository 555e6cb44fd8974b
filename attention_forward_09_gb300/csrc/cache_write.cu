// cache_write.cu -- KV cache write through slot_mapping for sm_103a.
//
// Operation: vllm-ascend attention_v1.py, AscendAttentionBackendImpl.
// reshape_and_cache -- each new token's key and value rows go into the paged
// cache (2, num_blocks, block_size, Hkv, D) at the token's slot, slot =
// block * block_size + offset (the AscendMetadata slot_mapping comment); a
// negative slot (a padding token) stores nothing.
//
// The copy is HBM-bound: 2 * Hkv * D * 2 bytes read and written per token.
// A token's [Hkv, D] row is contiguous both in key / value and in the cache
// (cache row = half * num_blocks * block_size + slot), so one warp copies one
// (token, K or V) row with 16-byte loads and stores, several in flight per
// lane; warps stride over the 2 * num_tokens rows.
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {  // read once: keep it out of L1
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__global__ void __launch_bounds__(256) kv_cache_write_sm103a(const CacheWriteParams p) {
    constexpr int kUnroll = 4;
    const int lane = threadIdx.x & 31;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < 2 * p.num_tokens;
         w += nwarps) {
        const long long t = w >> 1;
        const int half = static_cast<int>(w & 1);  // 0: key, 1: value
        const int slot = p.slot_mapping[t];
        if (slot < 0) continue;  // padding token
        if (slot >= p.num_slots) {
            if (lane == 0 && half == 0 && p.status) atomicOr(p.status, kDevBadIndex);
            continue;
        }
        const uint4* src = (half ? p.value : p.key) + t * p.row_vec;
        uint4* dst = p.cache + (static_cast<long long>(half) * p.num_slots + slot) * p.row_vec;
        for (int i0 = lane; i0 < p.row_vec; i0 += 32 * kUnroll) {
            uint4 r[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (i0 + 32 * u < p.row_vec) r[u] = ld_stream(src + i0 + 32 * u);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (i0 + 32 * u < p.row_vec) dst[i0 + 32 * u] = r[u];
        }
    }
}

cudaError_t launch_cache_write(const CacheWriteParams& p, int num_sms, cudaStream_t stream) {
    if (p.num_tokens <= 0) return cudaSuccess;
    const long long rows = 2 * p.num_tokens, warps_per_cta = 8;
    long long grid = (rows + warps_per_cta - 1) / warps_per_cta;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;  // 8 CTAs of 8 warps per SM
    if (grid > cap) grid = cap;
    kv_cache_write_sm103a<<<static_cast<unsigned>(grid), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gbattn
