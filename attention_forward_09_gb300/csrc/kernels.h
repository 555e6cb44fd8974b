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
    int linear;     // 1: blockIdx.x counts items from item_base; 2: persistent walk of packed documents
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
    // 1: every pipeline wait gives up at once (attn_set_wait_give_up, a test
    // of the failure path).  Set by the host API.
    int give_up;
    // Padded batch (dense mode only, attn_fwd_padded): batch entry b uses its
    // first lens_q[b] query rows and lens_k[b] keys (null: all of them).
    const int32_t* lens_q;
    const int32_t* lens_k;
};

// The give-up setting the host API passes to the prefill kernels (process-wide).
int prefill_give_up();

// Tensor maps are built by the host (api.cpp) over q [Tq, Hq, D] and
// k / v [Tk, Hkv, D] (box {64, 1, rows}) and over out [Tq, Hq, D] (box
// {128 bytes of columns, 1, 128}), all with 128-byte swizzle.
cudaError_t launch_prefill(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmO, const PrefillParams& p, int num_sms, cudaStream_t stream);
int prefill_block_n(int D);    // keys per KV tile for head size D
int prefill_v_box_rows(int D); // rows of the V map's TMA box for head size D

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


// Block-sparse video attention (vsa.cu).  The tiled layout holds block b of
// the sequence at rows [64 b, 64 b + 64), its first sizes[b] rows real, for
// nbp = nb rounded up to even blocks: tile t (128 rows) is query blocks 2 t
// and 2 t + 1, the second an empty partner when nb is odd.
constexpr int kVsaBlock = 64;

// A key-block entry of a tile's list: (block << 9) | (its token count << 2)
// | bits, bit 0 set when query block 2 t keeps the block, bit 1 when 2 t + 1
// does.  A list holds the blocks with bits 3, then 1, then 2, each group in
// ascending block order.
__host__ __device__ inline int vsa_entry(int blk, int size, int bits) { return (blk << 9) | (size << 2) | bits; }

// Sizes of the per-head list array: tile t holds up to capacity(t) entries
// from offset(t) on.  Tiles with a prefix query block (or every tile, when
// topk keeps every video block) list every block; the others at most the
// prefix blocks plus topk video blocks from each of their two query blocks.
struct VsaGeom {
    int nb, nt, n_prefix, keep, td, c2;
    __host__ __device__ static VsaGeom make(int nb_, int n_prefix_, int topk) {
        VsaGeom g;
        g.nb = nb_;
        g.nt = (nb_ + 1) / 2;
        g.n_prefix = n_prefix_;
        const int n_video = nb_ - n_prefix_;
        g.keep = topk < 0 ? 0 : (topk < n_video ? topk : n_video);
        const int dense_tiles = (n_prefix_ + 1) / 2;
        g.td = g.keep == n_video ? g.nt : (dense_tiles < g.nt ? dense_tiles : g.nt);
        const long long c2 = static_cast<long long>(n_prefix_) + 2LL * g.keep;
        g.c2 = c2 < nb_ ? static_cast<int>(c2) : nb_;
        return g;
    }
    __host__ __device__ int capacity(int t) const { return t < td ? nb : c2; }
    __host__ __device__ long long offset(int t) const {
        return t < td ? static_cast<long long>(t) * nb
                      : static_cast<long long>(td) * nb + static_cast<long long>(t - td) * c2;
    }
    __host__ __device__ long long per_head() const { return offset(nt); }
};

struct VsaFwdParams {
    void* out;                 // [out_rows, Hq, D]
    float* lse;                // [Hq, out_rows] or null
    uint32_t* status;
    const int32_t* kv_list;    // [Hq, g.per_head()]
    const int32_t* kv_num;     // [Hq, g.nt]
    const int32_t* out_index;  // [nbp * 64]: out row of each tiled row, -1 = none; null = identity
    long long out_rows;
    VsaGeom g;
    int Hq, group;
    float scale_log2;
    int out_f32;
};

// dst[w] = src[index[w]] for 0 <= index[w] < src_rows, zeros for a negative
// index; a larger one is flagged (kDevBadIndex) and zeroed.  row_bytes % 16 == 0.
cudaError_t launch_gather_rows(const void* src, long long src_rows, const int32_t* index, long long dst_rows,
                               int row_bytes, void* dst, uint32_t* status, int num_sms, cudaStream_t st);
// pooled [H, nb, D] fp32 = block means of the tiled x [nb * 64, H, D] bf16.
cudaError_t launch_vsa_pool(const void* x, const int32_t* sizes, int nb, int H, int D, float* pooled,
                            uint32_t* status, int num_sms, cudaStream_t st);
// Shared memory of the block-map kernel for qb query blocks per CTA, or -1 if over the limit.
int vsa_map_smem_bytes(int nb, int D, int qb);
cudaError_t launch_vsa_block_map(const float* pq, const float* pk, const int32_t* sizes, const VsaGeom& g, int Hq,
                                 int group, int D, float scale, int32_t* kv_list, int32_t* kv_num, uint32_t* status,
                                 cudaStream_t st);
// Tensor maps over the tiled q [nbp * 64, Hq, D] (box rows 128) and k / v
// [nbp * 64, Hkv, D] (box rows 64), box {64 columns, 1, rows}, 128-byte swizzle.
cudaError_t launch_vsa_fwd(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const VsaFwdParams& p, cudaStream_t st);

}  // namespace gbattn
