// masks.cu -- padding mask -> packed varlen documents and back, for sm_103a.
//
// Operation: vllm-omni flash_attn.py, FlashAttentionImpl._forward_varlen_masked
// -- a padded batch [B, S, H, D] with a [B, S] padding mask is packed (the
// masked-in tokens of each row, in order) into varlen documents, attended
// with cu_seqlens, and the output is put back at the tokens' positions with
// zeros at the padding.  Three memory-bound kernels, no host round trip:
//
//   mask_to_varlen   one CTA per batch row: cu_seqlens[b] is the number of
//                    masked-in tokens of rows < b (counted again by every CTA:
//                    B is small, the mask bytes come from L2), then a block
//                    scan of row b gives every token its packed row, or -1;
//   pack_rows        warp per row: x row (b, s) -> packed row pos[b*S + s];
//                    packed rows at or past the total are zeroed, so a varlen
//                    launch sized for B*S rows never reads uninitialised data;
//   unpack_rows      warp per padded row: the packed row, or zeros;
//   unpack_lse       lse [H, B*S packed] -> [B, H, S], -inf at the padding.
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {

// Block-wide exclusive prefix sum of one 0/1 flag per thread (blockDim.x =
// 1024); returns the prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int flag, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned ballot = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(ballot & ((1u << lane) - 1u));
    if (lane == 0) warp_sums[warp] = __popc(ballot);
    __syncthreads();
    if (warp == 0) {
        const int v = warp_sums[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        warp_sums[lane] = incl - v;  // exclusive, per warp
        if (lane == 31) *total = incl;
    }
    __syncthreads();
    const int r = warp_sums[warp] + in_warp;
    __syncthreads();  // warp_sums is reused by the next call
    return r;
}

__global__ void __launch_bounds__(1024) mask_to_varlen_sm103a(const uint8_t* mask, int B, int S, int32_t* cu_seqlens,
                                                              int32_t* packed_pos) {
    __shared__ int warp_sums[32];
    __shared__ int chunk_total;
    __shared__ int base_count;
    const int b = blockIdx.x;
    // masked-in tokens of rows < b
    int c = 0;
    for (long long i = threadIdx.x; i < static_cast<long long>(b) * S; i += blockDim.x) c += mask[i] != 0;
    c = __reduce_add_sync(0xffffffffu, c);
    if (threadIdx.x == 0) base_count = 0;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) atomicAdd(&base_count, c);
    __syncthreads();
    int run = base_count;
    if (threadIdx.x == 0) cu_seqlens[b] = run;
    const uint8_t* row = mask + static_cast<long long>(b) * S;
    int32_t* pos = packed_pos + static_cast<long long>(b) * S;
    for (int s0 = 0; s0 < S; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        const int flag = (s < S && row[s] != 0) ? 1 : 0;
        const int pre = block_exclusive_scan(flag, warp_sums, &chunk_total);
        if (s < S) pos[s] = flag ? run + pre : -1;
        run += chunk_total;
        __syncthreads();
    }
    if (b == B - 1 && threadIdx.x == 0) cu_seqlens[B] = run;
}

// Warp copy of one row of `vec` 16-byte vectors (or zeros when src is null).
__device__ __forceinline__ void warp_copy_row(uint4* dst, const uint4* src, int vec, int lane) {
    for (int i = lane; i < vec; i += 32) dst[i] = src ? src[i] : make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(256) pack_rows_sm103a(const uint4* x, const int32_t* packed_pos,
                                                        const int32_t* cu_seqlens, int B, long long rows, int vec,
                                                        uint4* packed) {
    const int lane = threadIdx.x & 31;
    const long long total = cu_seqlens[B];
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < 2 * rows; w += nw) {
        if (w < rows) {  // scatter row w to its packed row
            const int p = packed_pos[w];
            if (p >= 0 && p < rows) warp_copy_row(packed + p * static_cast<long long>(vec), x + w * vec, vec, lane);
        } else {         // packed rows past the total: zeros
            const long long p = w - rows;
            if (p >= total) warp_copy_row(packed + p * vec, nullptr, vec, lane);
        }
    }
}

__global__ void __launch_bounds__(256) unpack_rows_sm103a(const uint4* packed, const int32_t* packed_pos,
                                                          long long rows, int vec, uint4* out) {
    const int lane = threadIdx.x & 31;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < rows; w += nw) {
        const int p = packed_pos[w];
        warp_copy_row(out + w * vec, (p >= 0 && p < rows) ? packed + p * static_cast<long long>(vec) : nullptr, vec,
                      lane);
    }
}

__global__ void __launch_bounds__(256) unpack_lse_sm103a(const float* lse_packed, long long hstride,
                                                         const int32_t* packed_pos, int B, int H, int S, float* lse) {
    const long long n = static_cast<long long>(B) * H * S;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(i % S);
        const long long bh = i / S;
        const int h = static_cast<int>(bh % H), b = static_cast<int>(bh / H);
        const int p = packed_pos[static_cast<long long>(b) * S + s];
        lse[i] = p >= 0 ? lse_packed[h * hstride + p] : -INFINITY;
    }
}

static int copy_grid(long long warps, int num_sms) {
    long long g = (warps + 7) / 8;  // 8 warps per CTA
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;
    return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

cudaError_t launch_mask_to_varlen(const uint8_t* mask, int B, int S, int32_t* cu_seqlens, int32_t* packed_pos,
                                  cudaStream_t st) {
    mask_to_varlen_sm103a<<<B, 1024, 0, st>>>(mask, B, S, cu_seqlens, packed_pos);
    return cudaGetLastError();
}

cudaError_t launch_pack_rows(const void* x, const int32_t* packed_pos, const int32_t* cu_seqlens, int B, long long rows,
                             int row_bytes, void* packed, int num_sms, cudaStream_t st) {
    pack_rows_sm103a<<<copy_grid(2 * rows, num_sms), 256, 0, st>>>(static_cast<const uint4*>(x), packed_pos,
                                                                    cu_seqlens, B, rows, row_bytes / 16,
                                                                    static_cast<uint4*>(packed));
    return cudaGetLastError();
}

cudaError_t launch_unpack_rows(const void* packed, const int32_t* packed_pos, long long rows, int row_bytes, void* out,
                               int num_sms, cudaStream_t st) {
    unpack_rows_sm103a<<<copy_grid(rows, num_sms), 256, 0, st>>>(static_cast<const uint4*>(packed), packed_pos, rows,
                                                                 row_bytes / 16, static_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_unpack_lse(const float* lse_packed, long long hstride, const int32_t* packed_pos, int B, int H,
                              int S, float* lse, int num_sms, cudaStream_t st) {
    const long long n = static_cast<long long>(B) * H * S;
    long long g = (n + 255) / 256;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 16;
    unpack_lse_sm103a<<<static_cast<int>(g > cap ? cap : (g < 1 ? 1 : g)), 256, 0, st>>>(lse_packed, hstride,
                                                                                        packed_pos, B, H, S, lse);
    return cudaGetLastError();
}

}  // namespace gbattn
