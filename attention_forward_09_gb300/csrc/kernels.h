// kernels.h -- private interface between the host API and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gbattn {

constexpr uint32_t kDevBadIndex = 1u;
constexpr uint32_t kDevTimeout = 2u;
constexpr uint32_t kDevBadSeqlen = 4u;

// One launch of the prefill kernel.  Dense batches use cu_q == cu_k == nullptr
// and fixed lengths Sq / Sk per batch entry; packed documents use cu_seqlens.
struct PrefillParams {
    void* out;
    float* lse;
    uint32_t* status;
    const int32_t* cu_q;
    const int32_t* cu_k;
    int num_docs;      // B (dense) or number of documents
    int Sq, Sk;        // dense per-batch lengths
    int Tq, Tk;        // total rows of q and of k/v
    int max_seqlen_q;  // bound checked on the device
    int max_seqlen_k;
    int Hq, Hkv, group;
    float scale_log2;  // softmax_scale * log2(e)
    int causal;
    int out_f32;
    long long lse_bstride;  // lse offset = b*lse_bstride + h*lse_hstride + row
    long long lse_hstride;
    int lse_row_global;     // row counted from the start of the packed tensor (varlen)
    // Dense batches on the two-tile kernel use a 1D grid of items
    // (query tile, head, batch), tile fastest; varlen keeps the 3D grid
    // (tile, head, document).  Set by launch_prefill, not by callers.
    int linear;     // 1: blockIdx.x counts items from item_base
    int tiles;      // query tiles (2 x 128 rows) per (batch, head)
    int item_base;  // first item of this launch
    int split;      // > 1: each item is shared by a cluster of `split` CTAs, one key range each
    int persist;    // 1: CTA b walks items item_base + b + i * gridDim.x < item_end
    int item_end;
    // Prefill over the paged cache (block_table != nullptr; queries packed by
    // cu_q): K/V tile j of document s is cache block block_table[s *
    // max_blocks + j] (block size = BN = 128), Lk = seq_lens[s]; the K and V
    // maps both view the cache as {D, Hkv, 2 * num_blocks * 128}, V rows
    // num_blocks * 128 on.
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_blocks;
    int num_blocks;
    // GQA packing (cu_q modes, D <= 128): a CTA serves one KV head; a tile's
    // 128 rows are 128 / group tokens x the group's query heads (the Q and
    // out maps then have boxes {64 or 128 B, group, 128 / group}).
    int gqa_pack;
};

// Tensor maps are built by the host (api.cpp) over q [Tq, Hq, D] and
// k / v [Tk, Hkv, D] (box {64, 1, rows}) and over out [Tq, Hq, D] (box
// {128 bytes of columns, 1, 128}), all with 128-byte swizzle.
cudaError_t launch_prefill(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmO, const PrefillParams& p, int num_sms, cudaStream_t stream);
int prefill_block_n(int D);  // keys per KV tile for head size D

// How launch_prefill runs these sizes: kernel launches, items (CTAs of work),
// items launched whole, and the key split of the rest (0: none).
struct PrefillPlan {
    int launches;
    int split;
    int persist;  // the full-wave launch is persistent (one CTA per SM)
    int tiles;
    long long n_items;
    long long n_full;
};
cudaError_t prefill_plan(int D, const PrefillParams& p, int num_sms, PrefillPlan* plan);

struct PagedParams {
    const void* q;          // [S, Hq, D] bf16
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;
    float* lse;
    uint32_t* status;
    float* part_o;          // [S, Hq, max_splits, D]
    float* part_lse;        // [S, Hq, max_splits]
    int4* pairs;            // [S * max_splits] work list: (sequence, split, tok0, tok1), longest first
    int* sched;             // [0] work counter, [1] number of pairs (written by paged_schedule)
    int num_seqs, num_blocks, max_blocks_per_seq, max_seq_len;
    int Hq, Hkv, group, heads_per_cta;
    int blocks_per_split, max_splits;
    float scale_log2;
    int out_f32;
};

struct PagedPlan {
    int blocks_per_split;
    int max_splits;
    size_t o_bytes, lse_bytes, pairs_bytes;  // workspace sections, each 256-byte aligned
    size_t workspace_bytes;
};
PagedPlan paged_plan(int num_seqs, int Hq, int Hkv, int D, int max_seq_len);

int paged_slice_rows(int D);  // tokens per TMA box of the paged cache map

cudaError_t launch_paged(int D, const CUtensorMap& tmKV, const PagedParams& p, int num_sms,
                         cudaStream_t stream);

// KV cache write (cache_write.cu): key / value [T, Hkv, D] bf16 rows into the
// cache [2, num_blocks, block_size, Hkv, D] at slot_mapping[t].
struct CacheWriteParams {
    const uint4* key;
    const uint4* value;
    const int32_t* slot_mapping;
    uint4* cache;
    long long num_tokens;
    long long num_slots;  // num_blocks * block_size
    int row_vec;          // Hkv * D * 2 / 16: 16-byte vectors per token row
    uint32_t* status;
};
cudaError_t launch_cache_write(const CacheWriteParams& p, int num_sms, cudaStream_t stream);

// Padding mask <-> packed varlen (masks.cu).  mask [B, S] bytes (nonzero =
// token); cu_seqlens [B + 1]; packed_pos [B * S]: the token's packed row or -1.
cudaError_t launch_mask_to_varlen(const uint8_t* mask, int B, int S, int32_t* cu_seqlens, int32_t* packed_pos,
                                  cudaStream_t st);
// x [rows, row_bytes] -> packed [rows, row_bytes]; rows past cu_seqlens[B] zeroed
cudaError_t launch_pack_rows(const void* x, const int32_t* packed_pos, const int32_t* cu_seqlens, int B, long long rows,
                             int row_bytes, void* packed, int num_sms, cudaStream_t st);
// packed [rows, row_bytes] -> out [rows, row_bytes], zero rows where packed_pos < 0
cudaError_t launch_unpack_rows(const void* packed, const int32_t* packed_pos, long long rows, int row_bytes, void* out,
                               int num_sms, cudaStream_t st);
// lse_packed [H, hstride] -> lse [B, H, S], -inf where packed_pos < 0
cudaError_t launch_unpack_lse(const float* lse_packed, long long hstride, const int32_t* packed_pos, int B, int H,
                              int S, float* lse, int num_sms, cudaStream_t st);

}  // namespace gbattn
