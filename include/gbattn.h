/*
 * gbattn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * Every entry point computes, for each query row i of query head h,
 *
 *     out[i, h, :] = softmax_j(softmax_scale * q[i, h] . k[j, kv(h)]) @ v[j, kv(h)]
 *     lse[h, i]    = ln sum_j exp(softmax_scale * q[i, h] . k[j, kv(h)])
 *
 * over the keys j that row i may see, with kv(h) = h / (num_heads / num_kv_heads)
 * (GQA: consecutive query heads share one KV head).  The operation and its
 * argument set follow the attention backends of vllm-omni flash_attn.py
 * (FlashAttentionImpl: flash_attn_func / flash_attn_varlen_func routes, the
 * (out, lse) pair of _unwrap_flash_output) and vllm-ascend attention_v1.py
 * (AscendAttentionBackendImpl.forward_paged_attention over the paged cache).
 *
 * Conventions shared by all calls
 * -------------------------------
 *  - Inputs q, k, v and the KV cache are bfloat16, row-major, head_size
 *    contiguous.  head_size must be one of 64, 96, 128, 192, 256
 *    (FlashAttentionBackend.get_supported_head_sizes).
 *  - num_heads % num_kv_heads == 0 (AscendAttentionBackendImpl.__init__).
 *  - Causal masking is bottom-right aligned per document: key j is visible
 *    to query i iff j <= i + (Lk - Lq) (FlashAttentionImpl.forward_fa_npu).
 *    A row that sees no key gets out = 0 and lse = -inf.
 *  - softmax_scale must be finite and > 0; there is no implicit default.
 *  - The caller owns every buffer.  The library allocates nothing, never
 *    synchronises, and launches only on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).  All pointers named "device"
 *    must be device-accessible; q, k, v, kv_cache and out must be 16-byte
 *    aligned.
 *  - out is written in out_dtype (bf16 or fp32); lse is fp32 and optional
 *    (NULL = not written).
 *  - dev_status (optional, device uint32): kernels OR GBATTN_DEV_* bits into
 *    it when they meet bad indices or a timed-out wait; they never trap.  The
 *    caller zeroes it and reads it after synchronising.
 *  - Host-side validation failures return a status before anything is
 *    launched; GBATTN_ERR_CUDA reports a launch or driver error.
 *  - Only devices of compute capability 10.3 (GB300) are accepted.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GBATTN_OK = 0,
    GBATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale, Hq % Hkv != 0 */
    GBATTN_ERR_UNSUPPORTED = 2, /* head size, block size or output dtype not supported */
    GBATTN_ERR_ALIGNMENT = 3,   /* a tensor pointer is not 16-byte aligned */
    GBATTN_ERR_WORKSPACE = 4,   /* paged workspace missing or too small */
    GBATTN_ERR_CUDA = 5,        /* CUDA runtime / driver error (launch, attribute, tensor map) */
    GBATTN_ERR_DEVICE = 6,      /* current device is not compute capability 10.3 */
    GBATTN_ERR_SCRATCH_LIMIT = 7 /* attn_fwd_paged_noalloc: sizes need more than its built-in scratch */
} gbattn_status;

typedef enum {
    GBATTN_OUT_BF16 = 0,
    GBATTN_OUT_F32 = 1
} gbattn_dtype;

/* Bits the kernels OR into *dev_status. */
#define GBATTN_DEV_BAD_INDEX 1u   /* block_table entry, slot or row index out of range (skipped) */
#define GBATTN_DEV_TIMEOUT 2u     /* a pipeline wait gave up; that tile's output is invalid */
#define GBATTN_DEV_BAD_SEQLEN 4u  /* cu_seqlens / seq_lens inconsistent or above the stated max */

/*
 * attn_fwd_dense -- fixed-length batch (the flash_attn_func route of
 * FlashAttentionImpl.forward_cuda in vllm-omni flash_attn.py).
 *
 *   q    device bf16 [B, Sq, Hq, D]
 *   k, v device bf16 [B, Sk, Hkv, D]
 *   out  device [B, Sq, Hq, D] in out_dtype
 *   lse  device fp32 [B, Hq, Sq] or NULL
 *
 * Batch b attends only its own keys, and its result depends only on its own
 * rows of q, k and v (NaN or Inf in another batch entry does not reach it).
 * Equivalent to attn_fwd_varlen with
 * cu_seqlens_q = arange(0, (B+1)*Sq, Sq) and cu_seqlens_k likewise
 * (FlashAttentionImpl._flash_varlen_wrapper), except for the LSE layout.
 * B, Sq or Sk equal to 0 is allowed (Sk = 0 writes zeros and -inf; k and v
 * may then be NULL).
 */
gbattn_status attn_fwd_dense(const void* q, const void* k, const void* v,
                             int B, int Sq, int Sk, int Hq, int Hkv, int D,
                             float softmax_scale, int causal,
                             void* out, gbattn_dtype out_dtype, float* lse,
                             uint32_t* dev_status, void* stream);

/*
 * attn_fwd_padded -- a padded batch whose padding mask keeps each row's first
 * tokens (right padding): the case of FlashAttentionImpl._forward_varlen_masked
 * (vllm-omni flash_attn.py) where the unpad -> varlen -> pad pipeline of
 * attn_fwd_masked needs no packing, since each row's kept tokens already lie
 * together.  Results equal that pipeline's for such a mask.
 *
 *   q, k, v, out, lse  as for attn_fwd_dense ([B, Sq, Hq, D], [B, Sk, Hkv, D],
 *                      [B, Sq, Hq, D], [B, Hq, Sq])
 *   lens_q   device int32 [B] or NULL: batch entry b's queries are its first
 *            lens_q[b] rows (NULL: all Sq rows, the key-only mask of
 *            cross-attention)
 *   lens_k   device int32 [B] or NULL: its keys are its first lens_k[b] rows
 *            (NULL: all Sk)
 *
 * Query rows past lens_q[b] get out = 0 and lse = -inf; key and value rows
 * past lens_k[b] never reach a result, whatever they hold.  Causal masking is
 * bottom-right within the used lengths: query i of entry b sees key j iff
 * j <= i + lens_k[b] - lens_q[b].  A length outside [0, S] sets
 * GBATTN_DEV_BAD_SEQLEN and is clamped.  Host errors as for attn_fwd_dense.
 */
gbattn_status attn_fwd_padded(const void* q, const void* k, const void* v, const int32_t* lens_q,
                              const int32_t* lens_k, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                              float softmax_scale, int causal, void* out, gbattn_dtype out_dtype, float* lse,
                              uint32_t* dev_status, void* stream);

/*
 * attn_fwd_dense_plan -- how attn_fwd_dense runs these sizes on the current
 * device, for launch accounting and tests; it launches and allocates nothing
 * and has no counterpart on the pages.
 *   launches  out: kernel launches one attn_fwd_dense call makes (0 when
 *             B or Sq is 0)
 *   split     out: 0, or 2, 4 or 8 when the items of a partly filled last
 *             wave (non-causal, head size <= 128) are each shared by a
 *             cluster of that many CTAs along the keys
 * Errors: GBATTN_ERR_INVALID_ARG (null outputs, bad sizes),
 * GBATTN_ERR_UNSUPPORTED (head size), GBATTN_ERR_DEVICE / GBATTN_ERR_CUDA.
 */
gbattn_status attn_fwd_dense_plan(int B, int Sq, int Sk, int Hq, int Hkv, int D, int causal, int* launches,
                                  int* split);

/*
 * attn_fwd_varlen -- packed documents (FlashAttentionImpl._forward_varlen_packed,
 * flash_attn_varlen_func with cu_seqlens_q/k and max_seqlen_q/k).
 *
 *   q              device bf16 [Tq, Hq, D]
 *   k, v           device bf16 [Tk, Hkv, D]
 *   cu_seqlens_q/k device int32 [num_docs + 1]: 0 = c[0] <= c[1] <= ... <= c[N] <= Tq (Tk);
 *                  rows past c[N] belong to no document (never read into a result, never written)
 *   max_seqlen_q/k host ints, >= every document's length (they size the grid;
 *                  no device read happens on the host)
 *   out            device [Tq, Hq, D] in out_dtype
 *   lse            device fp32 [Hq, Tq] or NULL
 *
 * Document n owns query rows [cu_q[n], cu_q[n+1]) and key rows
 * [cu_k[n], cu_k[n+1]); no row attends across documents.  Empty documents
 * are allowed (with Tk = 0, k and v may be NULL).  A document longer than max_seqlen, or cu_seqlens that
 * decrease or run past Tq/Tk, set GBATTN_DEV_BAD_SEQLEN and that document's
 * rows are left unwritten.  A document's result depends only on its own
 * rows of q, k and v: the key and value rows past its end (the next
 * document's, or rows of k and v past cu_seqlens_k[N]) are never mixed in,
 * whatever they hold, NaN and Inf included.
 */
gbattn_status attn_fwd_varlen(const void* q, const void* k, const void* v,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                              int num_docs, int Tq, int Tk, int max_seqlen_q, int max_seqlen_k,
                              int Hq, int Hkv, int D, float softmax_scale, int causal,
                              void* out, gbattn_dtype out_dtype, float* lse,
                              uint32_t* dev_status, void* stream);

/*
 * attn_fwd_varlen_plan -- how many kernel launches attn_fwd_varlen makes for
 * these sizes on the current device (launch accounting and tests; it reads
 * no device memory, launches and allocates nothing, and has no counterpart
 * on the pages).  Arguments as for attn_fwd_varlen; launches is an output.
 */
gbattn_status attn_fwd_varlen_plan(int num_docs, int Tq, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                   int causal, int* launches);

/*
 * attn_fwd_paged_prefill -- several query tokens per sequence against the
 * paged cache: chunked prefill, prefill with a cache hit, speculative decode
 * (vllm-ascend attention_v1.py, AscendAttentionState PrefillCacheHit /
 * ChunkedPrefill / SpecDecoding, with the context read through block_table).
 *   q             device bf16 [Tq, Hq, D], sequences packed by cu_seqlens_q
 *   cu_seqlens_q  device int32 [num_seqs + 1]; sequence s owns query rows
 *                 [cu_seqlens_q[s], cu_seqlens_q[s + 1]), its last q_len_s
 *                 context tokens
 *   kv_cache, num_blocks, block_size (= 128), block_table,
 *   max_blocks_per_seq, seq_lens
 *                 as for attn_fwd_paged; seq_lens[s] counts the whole
 *                 context including the q_len_s new tokens, whose K/V must
 *                 already be in the cache (attn_kv_cache_write)
 *   max_seqlen_q  host int >= every q_len_s; max_seq_len host int >= every
 *                 seq_lens[s]
 *   causal        bottom-right: query i of sequence s sees keys
 *                 j <= i + seq_lens[s] - q_len_s
 *   out           device [Tq, Hq, D] in out_dtype; lse fp32 [Hq, Tq] or NULL
 * Cache slots past seq_lens[s] are never used, whatever they hold.  A
 * block_table entry outside [0, num_blocks) sets GBATTN_DEV_BAD_INDEX (the
 * sequence's result is then undefined); inconsistent cu_seqlens_q or
 * seq_lens set GBATTN_DEV_BAD_SEQLEN and the sequence is skipped.  Host
 * errors as for attn_fwd_varlen, plus GBATTN_ERR_UNSUPPORTED for
 * block_size != 128.
 */
gbattn_status attn_fwd_paged_prefill(const void* q, const void* kv_cache, int num_blocks, int block_size,
                                     const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                                     const int32_t* cu_seqlens_q, int num_seqs, int Tq, int max_seqlen_q,
                                     int max_seq_len, int Hq, int Hkv, int D, float softmax_scale, int causal,
                                     void* out, gbattn_dtype out_dtype, float* lse, uint32_t* dev_status,
                                     void* stream);

/*
 * Padding mask <-> packed documents, for padded batches (vllm-omni
 * flash_attn.py, FlashAttentionImpl._forward_varlen_masked: the masked-in
 * tokens of each row are packed in order, attended as varlen documents, and
 * the output goes back to their positions with zeros at the padding).  With
 * these helpers the whole path runs on the device with no host round trip:
 * attn_fwd_varlen is called with Tq = Tk = B * S rows and max_seqlen = S.
 *
 * attn_mask_to_varlen -- mask: device bytes [B, S], nonzero = token.
 *   cu_seqlens  out, device int32 [B + 1]: the packed document boundaries
 *   packed_pos  out, device int32 [B * S]: packed row of token (b, s), or -1
 *
 * attn_pack_rows -- x: device [B * S, row_bytes] (one token row each, e.g.
 *   Hkv * D bf16), packed: device [B * S, row_bytes].  Token (b, s) goes to
 *   packed row packed_pos[b * S + s]; rows at or past cu_seqlens[B] are
 *   zeroed, so that attention reads no uninitialised row.
 *
 * attn_unpack_rows -- packed [B * S, row_bytes] -> out [B * S, row_bytes]:
 *   the packed row of each token, zeros at the padding.
 *
 * attn_unpack_lse -- lse_packed fp32 [H, B * S] (attn_fwd_varlen's layout)
 *   -> lse fp32 [B, H, S], -inf at the padding.
 *
 * row_bytes must be a positive multiple of 16 and x, packed, out 16-byte
 * aligned.  Errors: GBATTN_ERR_INVALID_ARG, GBATTN_ERR_ALIGNMENT,
 * GBATTN_ERR_UNSUPPORTED (B * S >= 2^31), GBATTN_ERR_DEVICE / _CUDA.
 */
gbattn_status attn_mask_to_varlen(const uint8_t* mask, int B, int S, int32_t* cu_seqlens, int32_t* packed_pos,
                                  void* stream);
gbattn_status attn_pack_rows(const void* x, const int32_t* packed_pos, const int32_t* cu_seqlens, int B, int S,
                             int row_bytes, void* packed, void* stream);
gbattn_status attn_unpack_rows(const void* packed, const int32_t* packed_pos, int B, int S, int row_bytes, void* out,
                               void* stream);
gbattn_status attn_unpack_lse(const float* lse_packed, const int32_t* packed_pos, int B, int H, int S, float* lse,
                              void* stream);

/*
 * attn_vsa_layout -- host function (no device work): the token blocks of
 * block-sparse video attention (vllm-omni fastvideo_vsa.py,
 * _get_h3_tile_metadata).  The sequence is prefix_segments[0..num_segments)
 * tokens, each segment cut into chunks of `block` tokens, followed by a
 * T x H x W video grid (tokens in T, H, W order) cut into tile_t x tile_h x
 * tile_w boxes taken in T, H, W order, smaller at the grid's far edges
 * (the page: 4 x 4 x 4 boxes, blocks of 64).
 *   order        out, host int32 [total tokens]: token indices block by block
 *   block_start  out, host int32 [num_blocks + 1]: block b is
 *                order[block_start[b] .. block_start[b + 1])
 *   num_blocks, num_prefix_blocks  out
 * With order or block_start NULL only the counts are written (to size the
 * arrays).  Errors: GBATTN_ERR_INVALID_ARG (negative sizes, a box larger
 * than a block), GBATTN_ERR_UNSUPPORTED (more than 2^31 tokens).
 */
gbattn_status attn_vsa_layout(const int32_t* prefix_segments, int num_segments, int T, int H, int W, int tile_t,
                              int tile_h, int tile_w, int block, int32_t* order, int32_t* block_start,
                              int* num_blocks, int* num_prefix_blocks);

/*
 * attn_kv_cache_write -- store new tokens' keys and values into the paged
 * cache (vllm-ascend attention_v1.py, AscendAttentionBackendImpl.
 * reshape_and_cache; slot = block * block_size + offset, the AscendMetadata
 * slot_mapping comment).
 *   key, value    device bf16 [num_tokens, Hkv, D], row-major
 *   slot_mapping  device int32 [num_tokens]; token t goes to
 *                 kv_cache[0 (key) / 1 (value), slot / block_size,
 *                 slot % block_size, :, :]; a negative slot (padding token)
 *                 stores nothing
 *   kv_cache      device bf16 [2, num_blocks, block_size, Hkv, D], written in
 *                 place; only the slots named are touched
 *   block_size    any positive size (attn_fwd_paged reads 128)
 * Two tokens with the same slot: one of them is stored, which one is not
 * defined.  A slot >= num_blocks * block_size is skipped and sets
 * GBATTN_DEV_BAD_INDEX in dev_status.  Errors: GBATTN_ERR_INVALID_ARG,
 * GBATTN_ERR_UNSUPPORTED (head size; num_tokens >= 2^30, Hkv * D * 2 bytes
 * per row or num_blocks * block_size slots past 2^31 - 1),
 * GBATTN_ERR_ALIGNMENT (key, value, kv_cache not 16-byte aligned),
 * GBATTN_ERR_DEVICE / GBATTN_ERR_CUDA.
 */
gbattn_status attn_kv_cache_write(const void* key, const void* value, const int32_t* slot_mapping, int num_tokens,
                                  void* kv_cache, int num_blocks, int block_size, int Hkv, int D,
                                  uint32_t* dev_status, void* stream);

/*
 * attn_fwd_paged_workspace_size -- bytes of device workspace attn_fwd_paged
 * needs for these sizes (split-K partial results).  Pure host arithmetic; the
 * same arguments always give the same answer, so it can be queried once
 * before CUDA-graph capture (cf. the workspace query in
 * AscendAttentionBackendImpl.full_graph_pa).  Returns 0 for invalid sizes.
 */
size_t attn_fwd_paged_workspace_size(int num_seqs, int Hq, int Hkv, int D, int max_seq_len);

/*
 * attn_fwd_paged -- one query token per sequence over a paged KV cache
 * (AscendAttentionBackendImpl.forward_paged_attention; cache shape from
 * AscendAttentionBackend.get_kv_cache_shape).
 *
 *   q            device bf16 [num_seqs, Hq, D]
 *   kv_cache     device bf16 [2, num_blocks, block_size, Hkv, D]; [0] = keys, [1] = values
 *   block_size   must be 128 (AscendAttentionBackend.get_supported_block_size)
 *   block_table  device int32 [num_seqs, max_blocks_per_seq]; token t of
 *                sequence s lives in physical block block_table[s, t / 128],
 *                slot t % 128 (the slot_mapping rule of AscendMetadata).
 *                Entries past ceil(seq_lens[s] / 128) are never read.
 *   seq_lens     device int32 [num_seqs], each in [0, max_seq_len] and
 *                <= 128 * max_blocks_per_seq (context_lens)
 *   max_seq_len  host int bounding seq_lens (sizes the split-K grid)
 *   causal       accepted for symmetry; a single query sees its whole
 *                context under the bottom-right rule, so it has no effect
 *   out          device [num_seqs, Hq, D] in out_dtype
 *   lse          device fp32 [num_seqs, Hq] or NULL
 *   workspace    device buffer of at least
 *                attn_fwd_paged_workspace_size(num_seqs, Hq, Hkv, D, max_seq_len)
 *                bytes, 256-byte aligned; contents need no initialisation
 *
 * Slots of the last block past seq_len are never used.  A block_table
 * entry outside [0, num_blocks) sets GBATTN_DEV_BAD_INDEX and its tokens are
 * skipped; a seq_len above max_seq_len sets GBATTN_DEV_BAD_SEQLEN and is
 * clamped.  A sequence with seq_len 0 gets out = 0 and lse = -inf.
 */
gbattn_status attn_fwd_paged(const void* q, const void* kv_cache, int num_blocks, int block_size,
                             const int32_t* block_table, int max_blocks_per_seq,
                             const int32_t* seq_lens, int num_seqs, int max_seq_len,
                             int Hq, int Hkv, int D, float softmax_scale, int causal,
                             void* out, gbattn_dtype out_dtype, float* lse,
                             void* workspace, size_t workspace_bytes,
                             uint32_t* dev_status, void* stream);

/*
 * attn_fwd_paged_noalloc -- attn_fwd_paged for callers that cannot allocate
 * device memory when they run the decode (inside a CUDA-graph capture, where
 * cudaMalloc is not allowed; as a plugin in a framework that owns all device
 * memory; in a server whose memory budget is fixed at start-up).  The pages
 * have no counterpart of this call: it is an addition of this library.
 *
 * Same arguments and results as attn_fwd_paged, without workspace and
 * workspace_bytes.  The split-K scratch comes from one device array built
 * into the library, GBATTN_NOALLOC_SCRATCH_BYTES long, which every GPU that
 * has loaded the library's code holds until the process exits.
 *
 *  - Sizes needing more scratch than that (see attn_fwd_paged_workspace_size)
 *    are refused with GBATTN_ERR_SCRATCH_LIMIT before any CUDA call.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture on the device.  The address is kept for the
 *    life of the process: after cudaDeviceReset on a device the library's
 *    device code is loaded anew and the array may move, so do not call this
 *    entry point on that device again in the same process.
 *  - The call itself allocates nothing and frees nothing.
 *  - Every call on a device shares the same array, and the array keeps the
 *    previous call's contents (nothing in it needs to start at zero).  Calls
 *    that can overlap on the GPU (different streams without ordering between
 *    them) race on it and give wrong results: order them.
 */
#define GBATTN_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */
gbattn_status attn_fwd_paged_noalloc(const void* q, const void* kv_cache, int num_blocks, int block_size,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     const int32_t* seq_lens, int num_seqs, int max_seq_len,
                                     int Hq, int Hkv, int D, float softmax_scale, int causal,
                                     void* out, gbattn_dtype out_dtype, float* lse,
                                     uint32_t* dev_status, void* stream);

/*
 * attn_set_wait_give_up -- a switch for testing the failure path of the
 * prefill kernels (attn_fwd_dense, attn_fwd_varlen, attn_fwd_paged_prefill),
 * process-wide, for the launches made after the call.  on = 1: each CTA
 * gives up its pipeline waits at once, as if they had run out of time: it
 * issues no MMA, lets its copies land, frees its tensor memory, sets
 * GBATTN_DEV_TIMEOUT in dev_status and returns; the call comes back with
 * GBATTN_OK and the outputs undefined, and the context stays usable.  on = 0
 * (the default): waits give up only after one second, far above any
 * legitimate wait.  previous (may be NULL) receives the old setting.  No
 * counterpart on the pages (whose errors are raised, never rerouted:
 * fastvideo_vsa.py forward_cuda).  Errors: GBATTN_ERR_INVALID_ARG unless on
 * is 0 or 1.
 */
gbattn_status attn_set_wait_give_up(int on, int* previous);

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(gbattn_status status);

/*
 * Block-sparse video attention, device path (vllm-omni fastvideo_vsa.py,
 * _forward_h3 without the trained gate branch).  The steps, each a call:
 *
 *   attn_vsa_tile_map    (host) the tiled layout of a geometry;
 *   attn_gather_rows     q, k, v -> block-padded tiled q, k, v;
 *   attn_vsa_pool        block means of the tiled q and k (_pool_h3_tiles);
 *   attn_vsa_block_map   pooled scores -> the key blocks each query block
 *                        keeps (_build_h3_block_map), as per-tile lists;
 *   attn_fwd_vsa         block-sparse attention over those lists, each row
 *                        written back to its token's place.
 *
 * Tiled layout: nb blocks of at most 64 tokens (the layout of
 * attn_vsa_layout with 64-token blocks), padded to nbp = nb + (nb & 1)
 * blocks; block b occupies tiled rows [64 b, 64 b + 64), its first
 * block_sizes[b] rows real, the rest zero.  A tile is 128 rows: query blocks
 * 2 t and 2 t + 1 (the last an empty partner when nb is odd).
 *
 * attn_vsa_tile_map -- host function, arguments as attn_vsa_layout with
 *   64-token blocks (tile_t * tile_h * tile_w <= 64).
 *   tile_index   out, host int32 [nbp * 64]: token of each tiled row, -1 at
 *                padding rows
 *   block_sizes  out, host int32 [nb]: tokens of each block
 *   With tile_index or block_sizes NULL only the counts are written.
 *
 * attn_gather_rows -- dst[w] = src[index[w]] (rows of row_bytes bytes,
 *   a positive multiple of 16; src and dst 16-byte aligned device memory;
 *   index device int32 [dst_rows]).  A negative index gives a zero row; one
 *   at or past src_rows a zero row and GBATTN_DEV_BAD_INDEX.
 *
 * attn_vsa_pool -- x_tiled device bf16 [nb * 64 (or more), H, D]; pooled
 *   out, device fp32 [H, nb, D]: the mean of each block's real rows
 *   (pooled / block size, as the page divides by the true size).
 *   block_sizes device int32 [nb]; a size outside [0, 64] is clamped and
 *   sets GBATTN_DEV_BAD_INDEX.  pooled 16-byte aligned.
 *
 * attn_vsa_list_size -- host: *entries = the int32 count of the kv_list
 *   array for these sizes (all Hq heads).
 *
 * attn_vsa_block_map -- pooled_q fp32 [Hq, nb, D], pooled_k fp32 [Hkv, nb,
 *   D] (attn_vsa_pool's output), both 16-byte aligned.  Scores scale *
 *   pooled_q . pooled_k in fp32;
 *   a prefix query block (index < num_prefix_blocks) keeps every key block; a
 *   video query block keeps every prefix key block and its min(topk,
 *   nb - num_prefix_blocks) best video key blocks, ties to the lower block
 *   index (with topk >= the video block count every block is kept).  topk
 *   must be >= 1, as the page requires.
 *   kv_list  out, device int32 [attn_vsa_list_size entries]: per head h and
 *            tile t, the union of the key blocks that query blocks 2 t and
 *            2 t + 1 keep, each entry (block << 9) | (block size << 2) |
 *            bits, bit 0 set if block 2 t keeps it, bit 1 if 2 t + 1 does;
 *            the blocks both keep come first, then those only 2 t keeps,
 *            then those only 2 t + 1 keeps, each group ascending (any order
 *            is accepted by attn_fwd_vsa)
 *   kv_num   out, device int32 [Hq, (nb + 1) / 2]: entries of each list
 *   Placement: with keep = min(topk, nb - num_prefix_blocks), nt = (nb + 1)
 *   / 2, td = nt if keep == nb - num_prefix_blocks else min(nt,
 *   (num_prefix_blocks + 1) / 2) tiles that list every block, and c2 =
 *   min(nb, num_prefix_blocks + 2 keep), head h's lists start at h * E (E =
 *   the list size for Hq = 1) and tile t's at t * nb (t < td) or td * nb +
 *   (t - td) * c2, holding at most nb or c2 entries.
 *   Errors: GBATTN_ERR_UNSUPPORTED if the scores of two query blocks against
 *   every key block do not fit in shared memory (nb above about 21000);
 *   GBATTN_ERR_ALIGNMENT for a pooled array not 16-byte aligned.
 *
 * attn_fwd_vsa -- q_tiled [nbp * 64, Hq, D], k_tiled / v_tiled [nbp * 64,
 *   Hkv, D], device bf16, D = 64 or 128; the padding rows of a block (those
 *   past its token count) are never used, whatever they hold.  The real value
 *   rows of every key block in a tile's list enter the P.V product of both
 *   query blocks of the tile (with weight zero for the one that does not
 *   keep the block), so they must be finite.  kv_list / kv_num from
 *   attn_vsa_block_map with the same nb, num_prefix_blocks, topk and Hq.
 *   Row r of query block b attends the real rows of every key block its
 *   block keeps.  out_index device int32 [nbp * 64]: the out row of each
 *   tiled row (attn_vsa_tile_map's tile_index), -1 = not written; NULL writes
 *   out in the tiled layout (out_rows = nbp * 64).  out [out_rows, Hq, D]
 *   (bf16 or fp32), lse optional fp32 [Hq, out_rows]; a row that keeps no key
 *   gets out = 0, lse = -inf.  An entry naming a block outside [0, nb) or a
 *   list longer than its capacity sets GBATTN_DEV_BAD_INDEX, as does an
 *   out_index at or past out_rows (row skipped).
 *
 * Errors of the device calls: GBATTN_ERR_INVALID_ARG, GBATTN_ERR_UNSUPPORTED
 * (head size, more than 65535 tiles, heads x tiles above 2^31 - 1),
 * GBATTN_ERR_ALIGNMENT, GBATTN_ERR_DEVICE
 * / _CUDA.  None allocates or synchronises.
 */
gbattn_status attn_vsa_tile_map(const int32_t* prefix_segments, int num_segments, int T, int H, int W, int tile_t,
                                int tile_h, int tile_w, int32_t* tile_index, int32_t* block_sizes, int* num_blocks,
                                int* num_prefix_blocks);
gbattn_status attn_gather_rows(const void* src, long long src_rows, const int32_t* index, long long dst_rows,
                               int row_bytes, void* dst, uint32_t* dev_status, void* stream);
gbattn_status attn_vsa_pool(const void* x_tiled, int num_blocks, int H, int D, const int32_t* block_sizes,
                            float* pooled, uint32_t* dev_status, void* stream);
gbattn_status attn_vsa_list_size(int num_blocks, int num_prefix_blocks, int topk, int Hq, long long* entries);
gbattn_status attn_vsa_block_map(const float* pooled_q, const float* pooled_k, int num_blocks, int num_prefix_blocks,
                                 int Hq, int Hkv, int D, int topk, float softmax_scale, const int32_t* block_sizes,
                                 int32_t* kv_list, int32_t* kv_num, uint32_t* dev_status, void* stream);
gbattn_status attn_fwd_vsa(const void* q_tiled, const void* k_tiled, const void* v_tiled, int num_blocks,
                           int num_prefix_blocks, int topk, const int32_t* kv_list, const int32_t* kv_num,
                           const int32_t* out_index, long long out_rows, int Hq, int Hkv, int D, float softmax_scale,
                           void* out, gbattn_dtype out_dtype, float* lse, uint32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
