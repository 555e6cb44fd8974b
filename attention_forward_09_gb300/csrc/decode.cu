// decode.cu -- paged-KV decode (one query token per sequence) for sm_103a.
//
// Operation: vllm-ascend attention_v1.py, AscendAttentionBackendImpl.
// forward_paged_attention -- each sequence's query attends its whole context,
// read from the cache (2, num_blocks, 128, Hkv, D) through block_table and
// seq_lens (AscendAttentionBackend.get_kv_cache_shape; token t of sequence s
// is slot t % 128 of block block_table[s, t / 128], the AscendMetadata
// slot_mapping rule).
//
// The path is HBM-bound (about 4 bytes of K/V per multiply-add), so it runs on
// the CUDA cores, not the tensor cores:
//   * work item = (sequence, KV head, split of `blocks_per_split` blocks); a
//     persistent grid of one CTA per SM walks the items round-robin;
//   * one producer thread streams each 128-token block's K and V tile
//     (32 KB each at D = 128) with TMA into a ring of shared-memory slots, the
//     block id taken from block_table (bounds-checked; a bad id is skipped
//     and reported);
//   * 128 consumer threads: thread t scores token t against the GQA group's
//     query heads (each K byte is read once for the whole group), an online
//     softmax per head across the block, then O += P V with one thread per
//     (column pair, token group);
//   * each item writes a partial (o / l, lse); paged_combine merges the splits
//     with lse = ln sum_i exp(lse_i), o = sum_i exp(lse_i - lse) o_i.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {

constexpr int kBlk = 128;  // tokens per cache block
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D_, int HG_>
struct PagedCfg {
    static constexpr int D = D_;
    static constexpr int HG = HG_;                       // query heads per CTA (divides the GQA group)
    static constexpr int NCH = (D + 63) / 64;
    static constexpr int SLOT_BYTES = NCH * kBlk * 128;  // K or V of one block for one KV head
    static constexpr int STAGES = D <= 64 ? 8 : (D <= 128 ? 6 : (D <= 192 ? 4 : 3));
    static constexpr int DP = D / 2;                     // column pairs
    static constexpr int TG = DP <= 32 ? 4 : (DP <= 64 ? 2 : 1);  // token groups in P V
    static constexpr int TPG = kBlk / TG;                // tokens per group
    static constexpr int PV_THREADS = DP * TG;           // <= 128
    // shared memory: slots | q[HG][D] f32 | P[128][HG] f32 | red[2][4][HG] | acc[TG][HG][D] | flags | bars
    static constexpr int OFF_Q = STAGES * SLOT_BYTES;
    static constexpr int OFF_P = OFF_Q + HG * D * 4;
    static constexpr int OFF_RED = OFF_P + kBlk * HG * 4;
    static constexpr int OFF_ACC = OFF_RED + 2 * 4 * HG * 4;
    static constexpr int OFF_FLAG = OFF_ACC + TG * HG * D * 4;
    static constexpr int OFF_BAR = (OFF_FLAG + STAGES * 4 + 7) & ~7;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + 2 * STAGES * 8;
    static_assert(PV_THREADS <= 128, "P V thread map");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__device__ __forceinline__ void consumer_sync() {  // the 128 consumer threads only
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

struct ItemCoords {
    int s, kvh, h0, sp, b0, b1, L;
};

// Item `it` -> (sequence, head group, split); sp varies fastest so the splits
// of one long sequence land on different CTAs.
__device__ __forceinline__ ItemCoords item_coords(const PagedParams& p, int it, int n_hgroups,
                                                  uint32_t* status, bool report) {
    ItemCoords c;
    c.sp = it % p.max_splits;
    const int rest = it / p.max_splits;
    const int hg = rest % n_hgroups;
    c.s = rest / n_hgroups;
    const int per_kv = p.group / p.heads_per_cta;
    c.kvh = hg / per_kv;
    c.h0 = c.kvh * p.group + (hg % per_kv) * p.heads_per_cta;
    int L = p.seq_lens[c.s];
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * kBlk);
    if (L < 0 || L > cap) {
        if (report && status) atomicOr(status, kDevBadSeqlen);
        L = L < 0 ? 0 : cap;
    }
    c.L = L;
    const int nblk = (L + kBlk - 1) / kBlk;
    c.b0 = c.sp * p.blocks_per_split;
    c.b1 = min(nblk, c.b0 + p.blocks_per_split);
    return c;
}

template <class C>
__global__ void __launch_bounds__(160, 1)
    paged_decode_sm103a(const __grid_constant__ CUtensorMap tmKV, const PagedParams p) {
    constexpr int D = C::D, HG = C::HG, STAGES = C::STAGES, NCH = C::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sSlots = smem_u32(smem);
    float* sq = reinterpret_cast<float*>(smem + C::OFF_Q);    // [HG][D]
    float* sp_ = reinterpret_cast<float*>(smem + C::OFF_P);   // [128][HG]
    float* sred = reinterpret_cast<float*>(smem + C::OFF_RED);  // [2][4][HG]
    float* sacc = reinterpret_cast<float*>(smem + C::OFF_ACC);  // [TG][HG][D]
    volatile int* sflag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);  // slot holds a bad block
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    auto b_full = [&](int s) { return smem_u32(&bars[s]); };
    auto b_empty = [&](int s) { return smem_u32(&bars[STAGES + s]); };
    __shared__ int abort_flag_storage;
    volatile int* abort_flag = &abort_flag_storage;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int n_hgroups = p.Hkv * (p.group / p.heads_per_cta);
    const int n_items = p.num_seqs * n_hgroups * p.max_splits;

    if (status_has_timeout(p.status, kDevTimeout)) return;
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(b_full(s), 1);
            mbar_init(b_empty(s), 128);
        }
        abort_flag_storage = 0;
        fence_mbar_init();
    }
    __syncthreads();
    bool ok = true;

    if (warp == 4) {
        // --------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tmKV);
            int cnt = 0;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const ItemCoords c = item_coords(p, it, n_hgroups, p.status, false);
                for (int b = c.b0; ok && b < c.b1; ++b) {
                    const int blk = p.block_table[static_cast<long long>(c.s) * p.max_blocks_per_seq + b];
                    const bool valid = blk >= 0 && blk < p.num_blocks;
                    if (!valid && p.status) atomicOr(p.status, kDevBadIndex);
                    for (int kv = 0; kv < 2; ++kv, ++cnt) {
                        const int slot = cnt % STAGES, u = cnt / STAGES;
                        if (u > 0 && !(ok = mbar_wait(b_empty(slot), (u - 1) & 1, abort_flag))) {
                            *abort_flag = 1;
                            break;
                        }
                        sflag[slot] = valid ? 0 : 1;
                        if (valid) {
                            mbar_arrive_expect_tx(b_full(slot), C::SLOT_BYTES);
                            const int row = (kv * p.num_blocks + blk) * kBlk;
                            for (int ch = 0; ch < NCH; ++ch)
                                tma_load_3d(sSlots + slot * C::SLOT_BYTES + ch * kBlk * 128, &tmKV, b_full(slot),
                                            ch * 64, c.kvh, row);
                        } else {
                            mbar_arrive(b_full(slot));
                        }
                    }
                }
            }
            if (!ok) {
                // Drain: wait (bounded) for the copies still in flight.
                for (int t = (cnt > STAGES ? cnt - STAGES : 0); t < cnt; ++t)
                    mbar_wait_drain(b_full(t % STAGES), (t / STAGES) & 1);
            }
        }
    } else {
        // -------------------------------------------------------- consumers
        const float c2 = p.scale_log2;
        int cnt = 0;
        // P V thread map: column pair dp, token group tg.
        const bool pv_active = tid < C::PV_THREADS;
        const int dp = tid % C::DP, tg = tid / C::DP;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
            const ItemCoords c = item_coords(p, it, n_hgroups, p.status, tid == 0);
            if (c.b0 >= c.b1) continue;
            // this item's query heads -> shared f32
            consumer_sync();
            for (int e = tid; e < HG * D; e += 128) {
                const int i = e / D, d = e % D;
                const uint16_t* qh = reinterpret_cast<const uint16_t*>(p.q) +
                                     (static_cast<long long>(c.s) * p.Hq + c.h0 + i) * D + d;
                sq[e] = __uint_as_float(static_cast<uint32_t>(*qh) << 16);
            }
            consumer_sync();
            float m[HG], l[HG], acc[HG][2];
#pragma unroll
            for (int i = 0; i < HG; ++i) {
                m[i] = -INFINITY;
                l[i] = 0.f;
                acc[i][0] = acc[i][1] = 0.f;
            }
            for (int b = c.b0; b < c.b1; ++b) {
                const int nvalid = min(kBlk, c.L - b * kBlk);
                // ---------------- K: scores of token `tid` for the HG heads
                // A failed wait never leaves the loop: the consumers keep
                // meeting at the named barriers (which cannot time out) and
                // run through the remaining blocks on garbage, fast, because
                // every later wait sees the abort flag.
                int slot = cnt % STAGES;
                if (!mbar_wait(b_full(slot), (cnt / STAGES) & 1, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                }
                const bool bad = !ok || sflag[slot] != 0;
                float sc[HG];
#pragma unroll
                for (int i = 0; i < HG; ++i) sc[i] = 0.f;
                if (!bad && tid < nvalid) {
                    const uint32_t krow = sSlots + slot * C::SLOT_BYTES + tid * 128;
#pragma unroll
                    for (int pc = 0; pc < D / 8; ++pc) {
                        const uint32_t addr = krow + (pc >> 3) * kBlk * 128 + (((pc & 7) ^ (tid & 7)) << 4);
                        uint32_t k0, k1, k2, k3;
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(k0), "=r"(k1), "=r"(k2), "=r"(k3)
                                     : "r"(addr));
                        const float kf[8] = {bf_lo(k0), bf_hi(k0), bf_lo(k1), bf_hi(k1),
                                             bf_lo(k2), bf_hi(k2), bf_lo(k3), bf_hi(k3)};
#pragma unroll
                        for (int i = 0; i < HG; ++i) {
                            const float4 qa = *reinterpret_cast<const float4*>(sq + i * D + pc * 8);
                            const float4 qb = *reinterpret_cast<const float4*>(sq + i * D + pc * 8 + 4);
                            float a = sc[i];
                            a = fmaf(qa.x, kf[0], a);
                            a = fmaf(qa.y, kf[1], a);
                            a = fmaf(qa.z, kf[2], a);
                            a = fmaf(qa.w, kf[3], a);
                            a = fmaf(qb.x, kf[4], a);
                            a = fmaf(qb.y, kf[5], a);
                            a = fmaf(qb.z, kf[6], a);
                            a = fmaf(qb.w, kf[7], a);
                            sc[i] = a;
                        }
                    }
                }
                mbar_arrive(b_empty(slot));
                ++cnt;
                const bool live = !bad && tid < nvalid;
                // ---------------- online softmax across the block, per head
#pragma unroll
                for (int i = 0; i < HG; ++i) {
                    float v = live ? sc[i] * c2 : -INFINITY;
                    sc[i] = v;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    if (lane == 0) sred[warp * HG + i] = v;
                }
                consumer_sync();
                float alpha[HG];
#pragma unroll
                for (int i = 0; i < HG; ++i) {
                    const float bm = fmaxf(fmaxf(sred[i], sred[HG + i]), fmaxf(sred[2 * HG + i], sred[3 * HG + i]));
                    const float mn = fmaxf(m[i], bm);
                    alpha[i] = (mn == -INFINITY) ? 1.f : ex2(m[i] - mn);
                    const float msub = (mn == -INFINITY) ? 0.f : mn;
                    m[i] = mn;
                    float pv = ex2(sc[i] - msub);  // 0 for masked tokens
                    sp_[tid * HG + i] = pv;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) pv += __shfl_xor_sync(0xffffffffu, pv, o);
                    if (lane == 0) sred[4 * HG + warp * HG + i] = pv;
                }
                consumer_sync();
#pragma unroll
                for (int i = 0; i < HG; ++i)
                    l[i] = l[i] * alpha[i] + (sred[4 * HG + i] + sred[5 * HG + i]) + (sred[6 * HG + i] + sred[7 * HG + i]);
                // ---------------- V: O += P V
                slot = cnt % STAGES;
                if (!mbar_wait(b_full(slot), (cnt / STAGES) & 1, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                }
                if (pv_active) {
#pragma unroll
                    for (int i = 0; i < HG; ++i) {
                        acc[i][0] *= alpha[i];
                        acc[i][1] *= alpha[i];
                    }
                    if (!bad && ok) {
                        const int t0 = tg * C::TPG, t1 = min(t0 + C::TPG, nvalid);
                        const int d = 2 * dp, ch = d >> 6, byte = (d & 63) * 2;
                        const uint32_t vbase = sSlots + slot * C::SLOT_BYTES + ch * kBlk * 128 + (byte & 15);
                        const int piece = byte >> 4;
                        for (int t = t0; t < t1; ++t) {
                            uint32_t vv;
                            asm volatile("ld.shared.b32 %0, [%1];"
                                         : "=r"(vv)
                                         : "r"(vbase + t * 128 + ((piece ^ (t & 7)) << 4)));
                            const float v0 = bf_lo(vv), v1 = bf_hi(vv);
                            if constexpr (HG % 4 == 0) {
#pragma unroll
                                for (int i = 0; i < HG; i += 4) {
                                    const float4 pp = *reinterpret_cast<const float4*>(sp_ + t * HG + i);
                                    acc[i][0] = fmaf(pp.x, v0, acc[i][0]);
                                    acc[i][1] = fmaf(pp.x, v1, acc[i][1]);
                                    acc[i + 1][0] = fmaf(pp.y, v0, acc[i + 1][0]);
                                    acc[i + 1][1] = fmaf(pp.y, v1, acc[i + 1][1]);
                                    acc[i + 2][0] = fmaf(pp.z, v0, acc[i + 2][0]);
                                    acc[i + 2][1] = fmaf(pp.z, v1, acc[i + 2][1]);
                                    acc[i + 3][0] = fmaf(pp.w, v0, acc[i + 3][0]);
                                    acc[i + 3][1] = fmaf(pp.w, v1, acc[i + 3][1]);
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < HG; ++i) {
                                    const float pp = sp_[t * HG + i];
                                    acc[i][0] = fmaf(pp, v0, acc[i][0]);
                                    acc[i][1] = fmaf(pp, v1, acc[i][1]);
                                }
                            }
                        }
                    }
                }
                mbar_arrive(b_empty(slot));
                ++cnt;
                consumer_sync();  // P and the reduction scratch are rewritten by the next block
            }
            // ---------------- partial result of this item
            if (pv_active) {
#pragma unroll
                for (int i = 0; i < HG; ++i) {
                    sacc[(tg * HG + i) * D + 2 * dp] = acc[i][0];
                    sacc[(tg * HG + i) * D + 2 * dp + 1] = acc[i][1];
                }
            }
            consumer_sync();
            for (int e = tid; e < HG * D; e += 128) {
                const int i = e / D, d = e % D;
                float a = 0.f;
#pragma unroll
                for (int g = 0; g < C::TG; ++g) a += sacc[(g * HG + i) * D + d];
                const long long row = (static_cast<long long>(c.s) * p.Hq + c.h0 + i) * p.max_splits + c.sp;
                p.part_o[row * D + d] = l[i] > 0.f ? a / l[i] : 0.f;
                if (d == 0) p.part_lse[row] = l[i] > 0.f ? (m[i] + __log2f(l[i])) * kLn2f : -INFINITY;
            }
        }
    }
    if (!ok) {
        *abort_flag = 1;
        if (p.status) atomicOr(p.status, kDevTimeout);
    }
    __syncthreads();
}

// Merge the split partials of each (sequence, query head).
__global__ void __launch_bounds__(128) paged_combine(const PagedParams p, int D) {
    const int s = blockIdx.x / p.Hq, h = blockIdx.x % p.Hq;
    int L = p.seq_lens[s];
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * kBlk);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int nblk = (L + kBlk - 1) / kBlk;
    const int nsp = (nblk + p.blocks_per_split - 1) / p.blocks_per_split;
    const long long row0 = (static_cast<long long>(s) * p.Hq + h) * p.max_splits;
    float mx = -INFINITY;
    for (int i = 0; i < nsp; ++i) mx = fmaxf(mx, p.part_lse[row0 + i]);
    float wsum = 0.f;
    for (int i = 0; i < nsp; ++i) wsum += (mx == -INFINITY) ? 0.f : ex2((p.part_lse[row0 + i] - mx) * kLog2e);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const long long orow = static_cast<long long>(s) * p.Hq + h;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float a = 0.f;
        for (int i = 0; i < nsp; ++i) {
            const float w = (mx == -INFINITY) ? 0.f : ex2((p.part_lse[row0 + i] - mx) * kLog2e);
            a = fmaf(w, p.part_o[(row0 + i) * D + d], a);
        }
        a *= inv;
        if (p.out_f32)
            reinterpret_cast<float*>(p.out)[orow * D + d] = a;
        else
            reinterpret_cast<uint16_t*>(p.out)[orow * D + d] = static_cast<uint16_t>(pack_bf16x2(a, 0.f) & 0xFFFFu);
    }
    if (threadIdx.x == 0 && p.lse) p.lse[orow] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

// ------------------------------------------------------------------ host side
PagedPlan paged_plan(int num_seqs, int Hq, int Hkv, int D, int max_seq_len) {
    PagedPlan pl{1, 0, 0};
    if (num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_seq_len <= 0) return pl;
    const long long maxblk = (max_seq_len + kBlk - 1) / kBlk;
    // Aim for >= ~1200 (sequence, KV head, split) items so a persistent grid
    // of one CTA per SM stays balanced; cap a split at 16 blocks (2048 tokens).
    const long long units = static_cast<long long>(num_seqs) * Hkv * maxblk;
    long long bps = units / 1216;
    bps = bps < 1 ? 1 : (bps > 16 ? 16 : bps);
    pl.blocks_per_split = static_cast<int>(bps);
    pl.max_splits = static_cast<int>((maxblk + bps - 1) / bps);
    const size_t rows = static_cast<size_t>(num_seqs) * Hq * pl.max_splits;
    const size_t o_bytes = (rows * D * 4 + 255) & ~size_t(255);
    const size_t l_bytes = (rows * 4 + 255) & ~size_t(255);
    pl.workspace_bytes = o_bytes + l_bytes;
    return pl;
}

template <class C>
static cudaError_t launch_paged_cfg(const CUtensorMap& tm, const PagedParams& p, int num_sms, cudaStream_t st) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_sm103a<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int n_hgroups = p.Hkv * (p.group / p.heads_per_cta);
    const long long n_items = static_cast<long long>(p.num_seqs) * n_hgroups * p.max_splits;
    const int grid = static_cast<int>(n_items < num_sms ? n_items : num_sms);
    paged_decode_sm103a<C><<<grid, 160, C::SMEM_BYTES, st>>>(tm, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    paged_combine<<<p.num_seqs * p.Hq, 128, 0, st>>>(p, C::D);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_paged_d(const CUtensorMap& tm, const PagedParams& p, int num_sms, cudaStream_t st) {
    switch (p.heads_per_cta) {
        case 1: return launch_paged_cfg<PagedCfg<D, 1>>(tm, p, num_sms, st);
        case 2: return launch_paged_cfg<PagedCfg<D, 2>>(tm, p, num_sms, st);
        case 4: return launch_paged_cfg<PagedCfg<D, 4>>(tm, p, num_sms, st);
        case 8: return launch_paged_cfg<PagedCfg<D, 8>>(tm, p, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_paged(int D, const CUtensorMap& tm, const PagedParams& p, int num_sms, cudaStream_t st) {
    switch (D) {
        case 64: return launch_paged_d<64>(tm, p, num_sms, st);
        case 96: return launch_paged_d<96>(tm, p, num_sms, st);
        case 128: return launch_paged_d<128>(tm, p, num_sms, st);
        case 192: return launch_paged_d<192>(tm, p, num_sms, st);
        case 256: return launch_paged_d<256>(tm, p, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbattn
