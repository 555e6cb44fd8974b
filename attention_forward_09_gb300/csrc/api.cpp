// api.cpp -- the extern "C" entry points of gbattn.h: argument validation,
// TMA tensor-map encoding and kernel launches.  No allocation, no
// synchronisation; every launch goes to the caller's stream.
#include "../../include/gbattn.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <atomic>
#include <mutex>

#include "kernels.h"

namespace {

using gbattn::PagedParams;
using gbattn::PagedPlan;
using gbattn::PrefillParams;

bool head_size_ok(int d) { return d == 64 || d == 96 || d == 128 || d == 192 || d == 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool scale_ok(float s) { return isfinite(s) && s > 0.f; }
constexpr float kLog2e = 1.4426950408889634f;

// ---- driver entry point for cuTensorMapEncodeTiled (no link against libcuda)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Per-device facts: compute capability 10.3 and the SM count.
struct DeviceInfo {
    bool ok;
    int sms;
};

gbattn_status device_info(DeviceInfo* out) {
    static DeviceInfo cache[64];
    static bool have[64];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GBATTN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return GBATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GBATTN_ERR_CUDA;
        cache[dev] = DeviceInfo{major == 10 && minor == 3, sms};
        have[dev] = true;
    }
    *out = cache[dev];
    return out->ok ? GBATTN_OK : GBATTN_ERR_DEVICE;
}

// Tensor [rows, heads, D] (D contiguous; bf16, or fp32 when f32) as a 3-D
// TMA map with box {128 bytes of D, 1, box_rows} and 128-byte swizzle;
// loads read out-of-range elements as zero, stores skip them.
bool encode_rows_heads_d(CUtensorMap* m, const void* base, long long rows, int heads, int d, int box_rows,
                         bool f32 = false, int box_heads = 1) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es, static_cast<cuuint64_t>(heads) * d * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(box_heads),
                         static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Shared by the dense and varlen entries: validation of what they have in common.
// k and v may be null only when there are no keys at all (has_keys == false).
gbattn_status check_common(const void* q, const void* k, const void* v, const void* out, int Hq, int Hkv, int D,
                           float scale, gbattn_dtype odt, bool has_keys) {
    if (!q || !out || (has_keys && (!k || !v))) return GBATTN_ERR_INVALID_ARG;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!scale_ok(scale)) return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (odt != GBATTN_OUT_BF16 && odt != GBATTN_OUT_F32) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GBATTN_ERR_ALIGNMENT;
    return GBATTN_OK;
}

gbattn_status run_prefill(const void* q, const void* k, const void* v, long long Tq, long long Tk, int D,
                          PrefillParams& p, cudaStream_t st) {
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    CUtensorMap tq, tk, tv, to;
    const int bn = gbattn::prefill_block_n(D);
    // With no keys at all no KV tile is ever loaded; point the K/V maps at q
    // so that they are still well-formed.
    const bool no_keys = Tk == 0;
    if (!encode_rows_heads_d(&tq, q, Tq, p.Hq, D, 128) ||
        !encode_rows_heads_d(&tk, no_keys ? q : k, no_keys ? Tq : Tk, no_keys ? p.Hq : p.Hkv, D, bn) ||
        !encode_rows_heads_d(&tv, no_keys ? q : v, no_keys ? Tq : Tk, no_keys ? p.Hq : p.Hkv, D,
                             gbattn::prefill_v_box_rows(D)) ||
        !encode_rows_heads_d(&to, p.out, Tq, p.Hq, D, 128, p.out_f32 != 0))
        return GBATTN_ERR_CUDA;
    return gbattn::launch_prefill(D, tq, tk, tv, to, p, di.sms, st) == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

// 1: the prefill kernels give up every pipeline wait (attn_set_wait_give_up).
std::atomic<int> g_give_up{0};

}  // namespace

int gbattn::prefill_give_up() { return g_give_up.load(std::memory_order_relaxed); }

extern "C" {

gbattn_status attn_set_wait_give_up(int on, int* previous) {
    if (on != 0 && on != 1) return GBATTN_ERR_INVALID_ARG;
    const int old = g_give_up.exchange(on);
    if (previous) *previous = old;
    return GBATTN_OK;
}

const char* attn_status_string(gbattn_status s) {
    switch (s) {
        case GBATTN_OK: return "ok";
        case GBATTN_ERR_INVALID_ARG: return "invalid argument";
        case GBATTN_ERR_UNSUPPORTED: return "unsupported head size, block size or dtype";
        case GBATTN_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
        case GBATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case GBATTN_ERR_CUDA: return "CUDA error";
        case GBATTN_ERR_DEVICE: return "device is not compute capability 10.3 (GB300)";
        case GBATTN_ERR_SCRATCH_LIMIT: return "sizes need more scratch than attn_fwd_paged_noalloc has built in";
        default: return "unknown status";
    }
}

gbattn_status attn_fwd_dense(const void* q, const void* k, const void* v, int B, int Sq, int Sk, int Hq, int Hkv,
                             int D, float softmax_scale, int causal, void* out, gbattn_dtype out_dtype, float* lse,
                             uint32_t* dev_status, void* stream) {
    gbattn_status s = check_common(q, k, v, out, Hq, Hkv, D, softmax_scale, out_dtype, Sk != 0);
    if (s != GBATTN_OK) return s;
    if (B < 0 || Sq < 0 || Sk < 0) return GBATTN_ERR_INVALID_ARG;
    if (B > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Sq > 0x7fffffffLL || static_cast<long long>(B) * Sk > 0x7fffffffLL)
        return GBATTN_ERR_UNSUPPORTED;  // row counts are 32-bit on the device
    if (B == 0 || Sq == 0) return GBATTN_OK;
    PrefillParams p{};
    p.give_up = gbattn::prefill_give_up();
    p.out = out;
    p.lse = lse;
    p.status = dev_status;
    p.cu_q = p.cu_k = nullptr;
    p.num_docs = B;
    p.Sq = Sq;
    p.Sk = Sk;
    p.Tq = B * Sq;
    p.Tk = B * Sk;
    p.max_seqlen_q = Sq;
    p.max_seqlen_k = Sk;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.scale_log2 = softmax_scale * kLog2e;
    p.causal = causal ? 1 : 0;
    p.out_f32 = out_dtype == GBATTN_OUT_F32;
    p.lse_bstride = static_cast<long long>(Hq) * Sq;
    p.lse_hstride = Sq;
    p.lse_row_global = 0;
    return run_prefill(q, k, v, static_cast<long long>(B) * Sq, static_cast<long long>(B) * Sk, D, p,
                       static_cast<cudaStream_t>(stream));
}

gbattn_status attn_fwd_padded(const void* q, const void* k, const void* v, const int32_t* lens_q,
                              const int32_t* lens_k, int B, int Sq, int Sk, int Hq, int Hkv, int D,
                              float softmax_scale, int causal, void* out, gbattn_dtype out_dtype, float* lse,
                              uint32_t* dev_status, void* stream) {
    gbattn_status s = check_common(q, k, v, out, Hq, Hkv, D, softmax_scale, out_dtype, Sk != 0);
    if (s != GBATTN_OK) return s;
    if (B < 0 || Sq < 0 || Sk < 0) return GBATTN_ERR_INVALID_ARG;
    if (B > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Sq > 0x7fffffffLL || static_cast<long long>(B) * Sk > 0x7fffffffLL)
        return GBATTN_ERR_UNSUPPORTED;  // row counts are 32-bit on the device
    if (B == 0 || Sq == 0) return GBATTN_OK;
    PrefillParams p{};
    p.give_up = gbattn::prefill_give_up();
    p.out = out;
    p.lse = lse;
    p.status = dev_status;
    p.cu_q = p.cu_k = nullptr;
    p.lens_q = lens_q;
    p.lens_k = lens_k;
    p.num_docs = B;
    p.Sq = Sq;
    p.Sk = Sk;
    p.Tq = B * Sq;
    p.Tk = B * Sk;
    p.max_seqlen_q = Sq;
    p.max_seqlen_k = Sk;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.scale_log2 = softmax_scale * kLog2e;
    p.causal = causal ? 1 : 0;
    p.out_f32 = out_dtype == GBATTN_OUT_F32;
    p.lse_bstride = static_cast<long long>(Hq) * Sq;
    p.lse_hstride = Sq;
    p.lse_row_global = 0;
    return run_prefill(q, k, v, static_cast<long long>(B) * Sq, static_cast<long long>(B) * Sk, D, p,
                       static_cast<cudaStream_t>(stream));
}

gbattn_status attn_fwd_dense_plan(int B, int Sq, int Sk, int Hq, int Hkv, int D, int causal, int* launches,
                                  int* split) {
    if (!launches || !split) return GBATTN_ERR_INVALID_ARG;
    *launches = 0;
    *split = 0;
    if (B < 0 || Sq < 0 || Sk < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (B > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (B == 0 || Sq == 0) return GBATTN_OK;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    PrefillParams p{};
    p.num_docs = B;
    p.Sq = Sq;
    p.Sk = Sk;
    p.max_seqlen_q = Sq;
    p.max_seqlen_k = Sk;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.causal = causal ? 1 : 0;
    gbattn::PrefillPlan pl;
    if (gbattn::prefill_plan(D, p, di.sms, &pl) != cudaSuccess) return GBATTN_ERR_CUDA;
    *launches = pl.launches;
    *split = pl.split;
    return GBATTN_OK;
}

gbattn_status attn_fwd_varlen_plan(int num_docs, int Tq, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                   int causal, int* launches) {
    if (!launches) return GBATTN_ERR_INVALID_ARG;
    *launches = 0;
    if (num_docs < 0 || Tq < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (num_docs > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (num_docs == 0 || Tq == 0 || max_seqlen_q == 0) return GBATTN_OK;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    int dummy = 0;
    PrefillParams p{};
    p.cu_q = p.cu_k = &dummy;  // only tested for presence: the plan reads no device memory
    p.num_docs = num_docs;
    p.Tq = Tq;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seqlen_k;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.causal = causal ? 1 : 0;
    gbattn::PrefillPlan pl;
    if (gbattn::prefill_plan(D, p, di.sms, &pl) != cudaSuccess) return GBATTN_ERR_CUDA;
    *launches = pl.launches;
    return GBATTN_OK;
}

gbattn_status attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_k, int num_docs, int Tq, int Tk, int max_seqlen_q,
                              int max_seqlen_k, int Hq, int Hkv, int D, float softmax_scale, int causal, void* out,
                              gbattn_dtype out_dtype, float* lse, uint32_t* dev_status, void* stream) {
    gbattn_status s = check_common(q, k, v, out, Hq, Hkv, D, softmax_scale, out_dtype, Tk != 0);
    if (s != GBATTN_OK) return s;
    if (!cu_seqlens_q || !cu_seqlens_k) return GBATTN_ERR_INVALID_ARG;
    if (num_docs < 0 || Tq < 0 || Tk < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return GBATTN_ERR_INVALID_ARG;
    if (max_seqlen_q > Tq || max_seqlen_k > Tk) return GBATTN_ERR_INVALID_ARG;
    if (num_docs > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (num_docs == 0 || Tq == 0 || max_seqlen_q == 0) return GBATTN_OK;
    PrefillParams p{};
    p.give_up = gbattn::prefill_give_up();
    p.out = out;
    p.lse = lse;
    p.status = dev_status;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.num_docs = num_docs;
    p.Sq = p.Sk = 0;
    p.Tq = Tq;
    p.Tk = Tk;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seqlen_k;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.scale_log2 = softmax_scale * kLog2e;
    p.causal = causal ? 1 : 0;
    p.out_f32 = out_dtype == GBATTN_OUT_F32;
    p.lse_bstride = 0;
    p.lse_hstride = Tq;
    p.lse_row_global = 1;
    return run_prefill(q, k, v, Tq, Tk, D, p, static_cast<cudaStream_t>(stream));
}

gbattn_status attn_kv_cache_write(const void* key, const void* value, const int32_t* slot_mapping, int num_tokens,
                                  void* kv_cache, int num_blocks, int block_size, int Hkv, int D,
                                  uint32_t* dev_status, void* stream) {
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || Hkv <= 0) return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    // The kernel counts the 2 * num_tokens (token, K or V) rows and a row's
    // 16-byte pieces in 32-bit integers.
    if (num_tokens >= (1 << 30) || static_cast<long long>(Hkv) * D * 2 > 0x7fffffffLL)
        return GBATTN_ERR_UNSUPPORTED;
    if (num_tokens == 0) return GBATTN_OK;
    if (!key || !value || !slot_mapping || !kv_cache) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(kv_cache)) return GBATTN_ERR_ALIGNMENT;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    gbattn::CacheWriteParams p{};
    p.key = static_cast<const uint4*>(key);
    p.value = static_cast<const uint4*>(value);
    p.slot_mapping = slot_mapping;
    p.cache = static_cast<uint4*>(kv_cache);
    p.num_tokens = num_tokens;
    p.num_slots = static_cast<long long>(num_blocks) * block_size;
    p.row_vec = Hkv * D * 2 / 16;
    p.status = dev_status;
    return gbattn::launch_cache_write(p, di.sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GBATTN_OK
                                                                                          : GBATTN_ERR_CUDA;
}

gbattn_status attn_fwd_paged_prefill(const void* q, const void* kv_cache, int num_blocks, int block_size,
                                     const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                                     const int32_t* cu_seqlens_q, int num_seqs, int Tq, int max_seqlen_q,
                                     int max_seq_len, int Hq, int Hkv, int D, float softmax_scale, int causal,
                                     void* out, gbattn_dtype out_dtype, float* lse, uint32_t* dev_status,
                                     void* stream) {
    gbattn_status s = check_common(q, kv_cache, kv_cache, out, Hq, Hkv, D, softmax_scale, out_dtype, true);
    if (s != GBATTN_OK) return s;
    if (!block_table || !seq_lens || !cu_seqlens_q) return GBATTN_ERR_INVALID_ARG;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0 || num_seqs < 0 || Tq < 0 || max_seqlen_q < 0 ||
        max_seq_len < 0 || max_seqlen_q > Tq)
        return GBATTN_ERR_INVALID_ARG;
    if (block_size != 128) return GBATTN_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (num_seqs == 0 || Tq == 0 || max_seqlen_q == 0) return GBATTN_OK;
    DeviceInfo di;
    s = device_info(&di);
    if (s != GBATTN_OK) return s;
    PrefillParams p{};
    p.give_up = gbattn::prefill_give_up();
    p.out = out;
    p.lse = lse;
    p.status = dev_status;
    p.cu_q = cu_seqlens_q;
    p.cu_k = nullptr;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.num_docs = num_seqs;
    p.Tq = Tq;
    p.Tk = 0;
    p.max_seqlen_q = max_seqlen_q;
    p.max_seqlen_k = max_seq_len;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.scale_log2 = softmax_scale * kLog2e;
    p.causal = causal ? 1 : 0;
    p.out_f32 = out_dtype == GBATTN_OUT_F32;
    p.lse_bstride = 0;
    p.lse_hstride = Tq;
    p.lse_row_global = 1;
    // D <= 128 with a GQA group dividing 128: one CTA per KV head, a tile's
    // rows are 128 / group tokens x the group's heads (each KV byte read once
    // per group; short query chunks fill the tile group times better).
    const int g = Hq / Hkv;
    p.gqa_pack = (D <= 128 && g >= 2 && 128 % g == 0) ? 1 : 0;
    const int box_heads = p.gqa_pack ? g : 1, box_rows = 128 / box_heads;
    CUtensorMap tq, tk, tv, to;
    const long long cache_rows = 2LL * num_blocks * 128;
    if (!encode_rows_heads_d(&tq, q, Tq, Hq, D, box_rows, false, box_heads) ||
        !encode_rows_heads_d(&tk, kv_cache, cache_rows, Hkv, D, 128) ||
        !encode_rows_heads_d(&tv, kv_cache, cache_rows, Hkv, D, gbattn::prefill_v_box_rows(D)) ||
        !encode_rows_heads_d(&to, out, Tq, Hq, D, box_rows, p.out_f32 != 0, box_heads))
        return GBATTN_ERR_CUDA;
    return gbattn::launch_prefill(D, tq, tk, tv, to, p, di.sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_mask_to_varlen(const uint8_t* mask, int B, int S, int32_t* cu_seqlens, int32_t* packed_pos,
                                  void* stream) {
    if (B < 0 || S < 0) return GBATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * S > 0x7fffffffLL || B > 0x7fffffff / 2) return GBATTN_ERR_UNSUPPORTED;
    if (B == 0) return GBATTN_OK;
    if (!mask || !cu_seqlens || (S > 0 && !packed_pos)) return GBATTN_ERR_INVALID_ARG;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    return gbattn::launch_mask_to_varlen(mask, B, S, cu_seqlens, packed_pos, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_pack_rows(const void* x, const int32_t* packed_pos, const int32_t* cu_seqlens, int B, int S,
                             int row_bytes, void* packed, void* stream) {
    if (B < 0 || S < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return GBATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * S > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    if (B == 0 || S == 0) return GBATTN_OK;
    if (!x || !packed_pos || !cu_seqlens || !packed) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(packed)) return GBATTN_ERR_ALIGNMENT;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    return gbattn::launch_pack_rows(x, packed_pos, cu_seqlens, B, static_cast<long long>(B) * S, row_bytes, packed,
                                    di.sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_unpack_rows(const void* packed, const int32_t* packed_pos, int B, int S, int row_bytes, void* out,
                               void* stream) {
    if (B < 0 || S < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return GBATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * S > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    if (B == 0 || S == 0) return GBATTN_OK;
    if (!packed || !packed_pos || !out) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(out)) return GBATTN_ERR_ALIGNMENT;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    return gbattn::launch_unpack_rows(packed, packed_pos, static_cast<long long>(B) * S, row_bytes, out, di.sms,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_unpack_lse(const float* lse_packed, const int32_t* packed_pos, int B, int H, int S, float* lse,
                              void* stream) {
    if (B < 0 || S < 0 || H <= 0) return GBATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * S > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    if (B == 0 || S == 0) return GBATTN_OK;
    if (!lse_packed || !packed_pos || !lse) return GBATTN_ERR_INVALID_ARG;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    return gbattn::launch_unpack_lse(lse_packed, static_cast<long long>(B) * S, packed_pos, B, H, S, lse, di.sms,
                                     static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

size_t attn_fwd_paged_workspace_size(int num_seqs, int Hq, int Hkv, int D, int max_seq_len) {
    if (Hkv <= 0 || Hq % Hkv != 0 || !head_size_ok(D)) return 0;
    return gbattn::paged_plan(num_seqs, Hq, Hkv, D, max_seq_len).workspace_bytes;
}

gbattn_status attn_fwd_paged(const void* q, const void* kv_cache, int num_blocks, int block_size,
                             const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                             int num_seqs, int max_seq_len, int Hq, int Hkv, int D, float softmax_scale,
                             int causal, void* out, gbattn_dtype out_dtype, float* lse, void* workspace,
                             size_t workspace_bytes, uint32_t* dev_status, void* stream) {
    (void)causal;  // one query token sees its whole context under the bottom-right rule
    if (!q || !kv_cache || !block_table || !seq_lens || !out) return GBATTN_ERR_INVALID_ARG;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || !scale_ok(softmax_scale)) return GBATTN_ERR_INVALID_ARG;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0 || num_seqs < 0 || max_seq_len < 0)
        return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (block_size != 128) return GBATTN_ERR_UNSUPPORTED;
    if (out_dtype != GBATTN_OUT_BF16 && out_dtype != GBATTN_OUT_F32) return GBATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return GBATTN_ERR_ALIGNMENT;
    if (2LL * num_blocks * 128 > 0x7FFFFFFFLL) return GBATTN_ERR_UNSUPPORTED;  // TMA row coordinate is int32
    if (num_seqs == 0) return GBATTN_OK;
    const int group = Hq / Hkv;
    const int hg = group % 8 == 0 ? 8 : (group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1));
    const PagedPlan plan = gbattn::paged_plan(num_seqs, Hq, Hkv, D, max_seq_len > 0 ? max_seq_len : 1);
    if (!workspace || workspace_bytes < plan.workspace_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return GBATTN_ERR_WORKSPACE;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    CUtensorMap tm;
    if (!encode_rows_heads_d(&tm, kv_cache, 2LL * num_blocks * 128, Hkv, D, gbattn::paged_slice_rows(D)))
        return GBATTN_ERR_CUDA;
    PagedParams p{};
    p.q = q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.lse = lse;
    p.status = dev_status;
    char* ws = static_cast<char*>(workspace);
    p.part_o = reinterpret_cast<float*>(ws);
    p.part_lse = reinterpret_cast<float*>(ws + plan.o_bytes);
    p.pairs = reinterpret_cast<int4*>(ws + plan.o_bytes + plan.lse_bytes);
    p.sched = reinterpret_cast<int*>(ws + plan.o_bytes + plan.lse_bytes + plan.pairs_bytes);
    p.num_seqs = num_seqs;
    p.num_blocks = num_blocks;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_seq_len = max_seq_len;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = group;
    p.heads_per_cta = hg;
    p.blocks_per_split = plan.blocks_per_split;
    p.max_splits = plan.max_splits;
    p.scale_log2 = softmax_scale * kLog2e;
    p.out_f32 = out_dtype == GBATTN_OUT_F32;
    return gbattn::launch_paged(D, tm, p, di.sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}


// ---------------------------------------------------------------- block-sparse video attention
gbattn_status attn_gather_rows(const void* src, long long src_rows, const int32_t* index, long long dst_rows,
                               int row_bytes, void* dst, uint32_t* dev_status, void* stream) {
    if (src_rows < 0 || dst_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return GBATTN_ERR_INVALID_ARG;
    if (dst_rows == 0) return GBATTN_OK;
    if (!index || !dst || (src_rows > 0 && !src)) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return GBATTN_ERR_ALIGNMENT;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    return gbattn::launch_gather_rows(src, src_rows, index, dst_rows, row_bytes, dst, dev_status, di.sms,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_vsa_pool(const void* x_tiled, int num_blocks, int H, int D, const int32_t* block_sizes,
                            float* pooled, uint32_t* dev_status, void* stream) {
    if (num_blocks < 0 || H <= 0) return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (num_blocks == 0) return GBATTN_OK;
    if (!x_tiled || !block_sizes || !pooled) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(x_tiled) || !aligned16(pooled)) return GBATTN_ERR_ALIGNMENT;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    return gbattn::launch_vsa_pool(x_tiled, block_sizes, num_blocks, H, D, pooled, dev_status, di.sms,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_vsa_list_size(int num_blocks, int num_prefix_blocks, int topk, int Hq, long long* entries) {
    if (!entries || num_blocks < 0 || num_prefix_blocks < 0 || num_prefix_blocks > num_blocks || topk < 1 || Hq <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (num_blocks >= (1 << 22)) return GBATTN_ERR_UNSUPPORTED;  // block index field of a list entry
    *entries = static_cast<long long>(Hq) * gbattn::VsaGeom::make(num_blocks, num_prefix_blocks, topk).per_head();
    return GBATTN_OK;
}

gbattn_status attn_vsa_block_map(const float* pooled_q, const float* pooled_k, int num_blocks, int num_prefix_blocks,
                                 int Hq, int Hkv, int D, int topk, float softmax_scale, const int32_t* block_sizes,
                                 int32_t* kv_list, int32_t* kv_num, uint32_t* dev_status, void* stream) {
    if (num_blocks < 0 || num_prefix_blocks < 0 || num_prefix_blocks > num_blocks || topk < 1)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || !scale_ok(softmax_scale)) return GBATTN_ERR_INVALID_ARG;
    if (!head_size_ok(D)) return GBATTN_ERR_UNSUPPORTED;
    if (num_blocks >= (1 << 22) || Hq > 65535) return GBATTN_ERR_UNSUPPORTED;
    if (num_blocks == 0) return GBATTN_OK;
    if (!pooled_q || !pooled_k || !block_sizes || !kv_list || !kv_num) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(pooled_q) || !aligned16(pooled_k)) return GBATTN_ERR_ALIGNMENT;
    if (gbattn::vsa_map_smem_bytes(num_blocks, D, 2) < 0) return GBATTN_ERR_UNSUPPORTED;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    const gbattn::VsaGeom g = gbattn::VsaGeom::make(num_blocks, num_prefix_blocks, topk);
    return gbattn::launch_vsa_block_map(pooled_q, pooled_k, block_sizes, g, Hq, Hq / Hkv, D, softmax_scale, kv_list,
                                        kv_num, dev_status, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

gbattn_status attn_fwd_vsa(const void* q_tiled, const void* k_tiled, const void* v_tiled, int num_blocks,
                           int num_prefix_blocks, int topk, const int32_t* kv_list, const int32_t* kv_num,
                           const int32_t* out_index, long long out_rows, int Hq, int Hkv, int D, float softmax_scale,
                           void* out, gbattn_dtype out_dtype, float* lse, uint32_t* dev_status, void* stream) {
    if (num_blocks < 0 || num_prefix_blocks < 0 || num_prefix_blocks > num_blocks || topk < 1 || out_rows < 0)
        return GBATTN_ERR_INVALID_ARG;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || !scale_ok(softmax_scale)) return GBATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GBATTN_ERR_UNSUPPORTED;
    if (out_dtype != GBATTN_OUT_BF16 && out_dtype != GBATTN_OUT_F32) return GBATTN_ERR_UNSUPPORTED;
    const long long nbp = num_blocks + (num_blocks & 1);
    const long long rows = nbp * gbattn::kVsaBlock;
    if (num_blocks >= (1 << 22) || nbp / 2 > 65535 || Hq > 65535 || static_cast<long long>(Hq) * (nbp / 2) > 0x7fffffffLL)
        return GBATTN_ERR_UNSUPPORTED;
    if (!out_index && out_rows != rows) return GBATTN_ERR_INVALID_ARG;
    if (num_blocks == 0) return GBATTN_OK;
    if (!q_tiled || !k_tiled || !v_tiled || !kv_list || !kv_num || !out) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(q_tiled) || !aligned16(k_tiled) || !aligned16(v_tiled) || !aligned16(out))
        return GBATTN_ERR_ALIGNMENT;
    DeviceInfo di;
    gbattn_status s = device_info(&di);
    if (s != GBATTN_OK) return s;
    CUtensorMap tq, tk, tv;
    if (!encode_rows_heads_d(&tq, q_tiled, rows, Hq, D, 128) ||
        !encode_rows_heads_d(&tk, k_tiled, rows, Hkv, D, gbattn::kVsaBlock) ||
        !encode_rows_heads_d(&tv, v_tiled, rows, Hkv, D, gbattn::kVsaBlock))
        return GBATTN_ERR_CUDA;
    gbattn::VsaFwdParams p{};
    p.out = out;
    p.lse = lse;
    p.status = dev_status;
    p.kv_list = kv_list;
    p.kv_num = kv_num;
    p.out_index = out_index;
    p.out_rows = out_rows;
    p.g = gbattn::VsaGeom::make(num_blocks, num_prefix_blocks, topk);
    p.Hq = Hq;
    p.group = Hq / Hkv;
    p.scale_log2 = softmax_scale * kLog2e;
    p.out_f32 = out_dtype == GBATTN_OUT_F32;
    return gbattn::launch_vsa_fwd(D, tq, tk, tv, p, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GBATTN_OK
               : GBATTN_ERR_CUDA;
}

}  // extern "C"
