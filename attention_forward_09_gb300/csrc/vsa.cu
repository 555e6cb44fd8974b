// vsa.cu -- block-sparse video attention for sm_103a.
//
// Operation: vllm-omni fastvideo_vsa.py, _forward_h3 without the trained gate
// branch.  The sequence (a prefix, then a T x H x W video latent grid) is cut
// into blocks of at most 64 tokens (_get_h3_tile_metadata); q, k and v are
// reordered into a block-padded "tiled" layout, block b at rows [64 b, 64 b +
// 64) with its first sizes[b] rows real; every block is mean-pooled
// (_pool_h3_tiles); pooled block scores scale * mean_q . mean_k pick, for each
// video query block, its topk best video key blocks plus every prefix key
// block, while prefix query blocks keep everything (_build_h3_block_map); and
// each query token attends the tokens of the key blocks its block keeps.
//
//   gather_rows      warp per destination row: dst[w] = src[index[w]] or zeros;
//   vsa_pool         thread per (block, head, 8 columns): fp32 block means;
//   vsa_block_map    CTA per (head, 8 / 4 / 2 query blocks): the pooled
//                    scores of those query blocks against every key block
//                    (fp32 FMA, two key blocks x 8 query blocks per thread)
//                    in shared memory, a 4-pass radix select of the topk-th score per
//                    query block (ties to the lower block index), and, per
//                    pair of query blocks, the union of their key blocks
//                    (kept by both, then by the first only, then the second);
//   vsa_fwd          CTA per (head, pair of query blocks = one 128-row tile):
//                    Q tile by TMA, K/V tiles of two 64-row key blocks taken
//                    from the pair's union list and loaded in the order the
//                    MMAs read them (K_0, K_1 V_0, K_2 V_1, ...), S = Q K^T and
//                    O += P V by tcgen05.mma with accumulators in TMEM, online
//                    softmax where each row masks the key blocks its own query
//                    block does not keep and the padding rows of every key
//                    block; P goes to TMEM columns of its own (two buffers)
//                    and is read from there by P V; a warp of its own zeroes
//                    the padding rows of each V tile once it has landed.
//
// The pair layout follows the page's note that the Blackwell kernel serves two
// 64-row query blocks per CTA (hence an even block count, the last block of an
// odd count being an empty partner).
#include <math.h>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {

// ------------------------------------------------------------------ gather
__global__ void __launch_bounds__(256) gather_rows_sm103a(const uint4* src, long long src_rows, const int32_t* index,
                                                          long long dst_rows, int vec, uint4* dst, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < dst_rows; w += nw) {
        long long i = index[w];
        if (i >= src_rows) {
            if (lane == 0 && status) atomicOr(status, kDevBadIndex);
            i = -1;
        }
        uint4* d = dst + w * vec;
        if (i >= 0) {
            const uint4* s = src + i * vec;
            for (int c = lane; c < vec; c += 32) d[c] = s[c];
        } else {
            for (int c = lane; c < vec; c += 32) d[c] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Token count of block b, clamped to [0, 64]; an out-of-range count is flagged.
__device__ __forceinline__ int block_size_at(const int32_t* sizes, int b, uint32_t* status) {
    int s = sizes[b];
    if (s < 0 || s > kVsaBlock) {
        if (status) atomicOr(status, kDevBadIndex);
        s = s < 0 ? 0 : kVsaBlock;
    }
    return s;
}

// -------------------------------------------------------------------- pool
// pooled[h][b][d] = (sum of rows r < sizes[b] of x[64 b + r][h][d]) / max(sizes[b], 1).
// Consecutive threads take consecutive 16-byte pieces of one token row.
__global__ void __launch_bounds__(256) vsa_pool_sm103a(const uint4* x, const int32_t* sizes, int nb, int H, int D,
                                                       float* pooled, uint32_t* status) {
    const int G = D / 8;
    const long long row_vec = static_cast<long long>(H) * G;
    const long long n = static_cast<long long>(nb) * row_vec;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int g = static_cast<int>(i % G);
        const long long bh = i / G;
        const int h = static_cast<int>(bh % H), b = static_cast<int>(bh / H);
        const int sz = block_size_at(sizes, b, g == 0 ? status : nullptr);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint4* src = x + static_cast<long long>(b) * kVsaBlock * row_vec + static_cast<long long>(h) * G + g;
#pragma unroll 4
        for (int r = 0; r < sz; ++r) {
            const uint4 v = src[r * row_vec];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[2 * e] += __uint_as_float(w[e] << 16);
                acc[2 * e + 1] += __uint_as_float(w[e] & 0xffff0000u);
            }
        }
        const float den = static_cast<float>(sz > 1 ? sz : 1);
        float4* dst = reinterpret_cast<float4*>(pooled + (static_cast<long long>(h) * nb + b) * D + g * 8);
        dst[0] = make_float4(acc[0] / den, acc[1] / den, acc[2] / den, acc[3] / den);
        dst[1] = make_float4(acc[4] / den, acc[5] / den, acc[6] / den, acc[7] / den);
    }
}

// --------------------------------------------------------------- block map
// Monotone map of a float onto uint32 (larger float, larger key); -0 counts as +0.
__device__ __forceinline__ uint32_t order_key(float s) {
    const uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct VsaMapParams {
    const float* pq;  // [Hq, nb, D]
    const float* pk;  // [Hkv, nb, D]
    const int32_t* sizes;
    int32_t* kv_list;
    int32_t* kv_num;
    uint32_t* status;
    VsaGeom g;
    int group, D, qb;
    float scale;
};

constexpr int kMapWarps = 8;
constexpr int kMapQB = 8;                     // most query blocks per CTA
constexpr int kMapKeys = 2 * kMapWarps * 32;  // key blocks per scoring pass (two per thread)
constexpr int kMapDC = 16;                    // dimensions per staged chunk of pooled keys
constexpr int kMapKS = kMapDC + 4;            // staged row stride in floats (conflict-free float4 reads)

__global__ void __launch_bounds__(kMapWarps * 32) vsa_block_map_sm103a(const VsaMapParams p) {
    extern __shared__ float4 map_smem[];
    const int QB = p.qb, D = p.D, nb = p.g.nb, n_prefix = p.g.n_prefix, keep = p.g.keep;
    const int words = (nb + 31) >> 5;
    float* pq_s = reinterpret_cast<float*>(map_smem);                  // [kMapQB][D]
    float* stage = pq_s + kMapQB * D;                                  // [kMapKeys][kMapKS]
    float* sc = stage + kMapKeys * kMapKS;                             // [QB][nb]
    uint32_t* sel = reinterpret_cast<uint32_t*>(sc + QB * nb);         // [QB][words] kept key blocks
    int* hist = reinterpret_cast<int*>(sel + QB * words);              // [kMapWarps][256]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, kvh = h / p.group;
    const int i0 = blockIdx.x * QB;

    for (int x = threadIdx.x; x < kMapQB * D; x += blockDim.x) {
        const int i = x / D;
        pq_s[x] = (i < QB && i0 + i < nb) ? p.pq[(static_cast<long long>(h) * nb + i0 + i) * D + x % D] : 0.f;
    }

    // Scores of the query blocks against every key block: thread t takes key
    // blocks kb + t and kb + t + 256 of each pass against all kMapQB query
    // blocks (16 fp32 sums in registers, each over d in ascending order); the
    // pooled keys pass through shared memory kMapDC dimensions at a time, the
    // pooled queries are read from there as broadcasts.
    const float* pkh = p.pk + static_cast<long long>(kvh) * nb * D;
    const int tid = threadIdx.x;
    for (int kb = 0; kb < nb; kb += kMapKeys) {
        float acc[2][kMapQB];
#pragma unroll
        for (int i = 0; i < kMapQB; ++i) acc[0][i] = acc[1][i] = 0.f;
        for (int d0 = 0; d0 < D; d0 += kMapDC) {
            __syncthreads();  // the previous chunk has been read (and pq_s written, the first time)
            for (int f = tid; f < kMapKeys * (kMapDC / 4); f += kMapWarps * 32) {
                const int key = f / (kMapDC / 4), c4 = f % (kMapDC / 4);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (kb + key < nb)
                    v = *reinterpret_cast<const float4*>(pkh + static_cast<long long>(kb + key) * D + d0 + 4 * c4);
                *reinterpret_cast<float4*>(stage + key * kMapKS + 4 * c4) = v;
            }
            __syncthreads();
#pragma unroll
            for (int dd = 0; dd < kMapDC; dd += 4) {
                const float4 k0 = *reinterpret_cast<const float4*>(stage + tid * kMapKS + dd);
                const float4 k1 = *reinterpret_cast<const float4*>(stage + (tid + kMapWarps * 32) * kMapKS + dd);
#pragma unroll
                for (int i = 0; i < kMapQB; ++i) {
                    const float4 q = *reinterpret_cast<const float4*>(pq_s + i * D + d0 + dd);
                    acc[0][i] = fmaf(q.x, k0.x, acc[0][i]);
                    acc[1][i] = fmaf(q.x, k1.x, acc[1][i]);
                    acc[0][i] = fmaf(q.y, k0.y, acc[0][i]);
                    acc[1][i] = fmaf(q.y, k1.y, acc[1][i]);
                    acc[0][i] = fmaf(q.z, k0.z, acc[0][i]);
                    acc[1][i] = fmaf(q.z, k1.z, acc[1][i]);
                    acc[0][i] = fmaf(q.w, k0.w, acc[0][i]);
                    acc[1][i] = fmaf(q.w, k1.w, acc[1][i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kMapQB; ++i) {
            if (i < QB) {
                if (kb + tid < nb) sc[i * nb + kb + tid] = p.scale * acc[0][i];
                if (kb + tid + kMapWarps * 32 < nb) sc[i * nb + kb + tid + kMapWarps * 32] = p.scale * acc[1][i];
            }
        }
    }
    __syncthreads();

    // kept key blocks of each query block (warp per query block)
    for (int qw = warp; qw < QB; qw += kMapWarps) {
        const int qi = i0 + qw;
        uint32_t* srow = sel + qw * words;
        const float* row = sc + qw * nb;
        if (qi >= nb) {
            for (int w = lane; w < words; w += 32) srow[w] = 0u;
        } else if (qi < n_prefix || keep == nb - n_prefix) {  // dense rows
            for (int w = lane; w < words; w += 32) {
                const int left = nb - w * 32;
                srow[w] = left >= 32 ? 0xffffffffu : ((1u << left) - 1u);
            }
        } else {
            // T = the keep-th largest key among the video key blocks, found
            // 8 bits at a time; need_eq = how many blocks with key T are kept.
            uint32_t T = 0xffffffffu;
            int need_eq = 0;
            if (keep > 0) {
                int* hs = hist + warp * 256;
                uint32_t prefix = 0u, pmask = 0u;
                int rem = keep;
                for (int shift = 24; shift >= 0; shift -= 8) {
                    for (int b = lane; b < 256; b += 32) hs[b] = 0;
                    __syncwarp();
                    for (int j = n_prefix + lane; j < nb; j += 32) {
                        const uint32_t k = order_key(row[j]);
                        if ((k & pmask) == prefix) atomicAdd(&hs[(k >> shift) & 255u], 1);
                    }
                    __syncwarp();
                    int c[8], s = 0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {  // lane l holds bins 255 - 8 l down to 248 - 8 l
                        c[e] = hs[255 - 8 * lane - e];
                        s += c[e];
                    }
                    int incl = s;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int v = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += v;
                    }
                    const uint32_t bal = __ballot_sync(0xffffffffu, incl >= rem);
                    const int L = bal ? __ffs(bal) - 1 : 31;
                    int bin = 0, above = 0;
                    if (lane == L) {
                        int acc = incl - s;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            if (acc + c[e] >= rem) {
                                bin = 255 - 8 * lane - e;
                                above = acc;
                                break;
                            }
                            acc += c[e];
                        }
                    }
                    bin = __shfl_sync(0xffffffffu, bin, L);
                    above = __shfl_sync(0xffffffffu, above, L);
                    rem -= above;
                    prefix |= static_cast<uint32_t>(bin) << shift;
                    pmask |= 0xffu << shift;
                    __syncwarp();
                }
                T = prefix;
                need_eq = rem;
            }
            int eq_before = 0;
            for (int base = 0; base < nb; base += 32) {
                const int j = base + lane;
                bool take = false, eq = false;
                if (j < nb) {
                    if (j < n_prefix) {
                        take = true;
                    } else if (keep > 0) {
                        const uint32_t k = order_key(row[j]);
                        take = k > T;
                        eq = k == T;
                    }
                }
                const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
                if (eq) take = eq_before + __popc(eqb & ((1u << lane) - 1u)) < need_eq;
                eq_before += __popc(eqb);
                const uint32_t tb = __ballot_sync(0xffffffffu, take);
                if (lane == 0) srow[base >> 5] = tb;
            }
        }
    }
    __syncthreads();

    // union list of each pair of query blocks (warp per pair; QB / 2 <= kMapWarps)
    if (warp < QB / 2) {
        const int t = (i0 >> 1) + warp;
        if (t < p.g.nt) {
            const uint32_t* s0 = sel + (2 * warp) * words;
            const uint32_t* s1 = s0 + words;
            int32_t* dst = p.kv_list + static_cast<long long>(h) * p.g.per_head() + p.g.offset(t);
            const int cap = p.g.capacity(t);
            // Blocks kept by both query blocks first, then those kept by the
            // first only, then by the second only: a K/V tile of two blocks
            // from one of the last two groups is skipped outright by the
            // softmax warps of the other query block.
            int cnt = 0;
#pragma unroll 1
            for (uint32_t want = 3u; want != 0u; want = want == 3u ? 1u : (want == 1u ? 2u : 0u)) {
                for (int w = 0; w < words; ++w) {
                    const int j = w * 32 + lane;
                    const uint32_t bits = ((s0[w] >> lane) & 1u) | (((s1[w] >> lane) & 1u) << 1);
                    const bool mine = bits == want;
                    const uint32_t sel_w = __ballot_sync(0xffffffffu, mine);
                    if (mine) {
                        const int at = cnt + __popc(sel_w & ((1u << lane) - 1u));
                        const int sz = block_size_at(p.sizes, j, p.status);
                        if (at < cap) dst[at] = vsa_entry(j, sz, static_cast<int>(bits));
                    }
                    cnt += __popc(sel_w);
                }
            }
            if (lane == 0) {
                if (cnt > cap && p.status) atomicOr(p.status, kDevBadIndex);
                p.kv_num[static_cast<long long>(h) * p.g.nt + t] = cnt < cap ? cnt : cap;
            }
        }
    }
}

// --------------------------------------------------------------- attention
template <int D_, int SLOTS_>
struct VsaCfg {
    static constexpr int D = D_;
    // Ring slots, each one load: K_{u} (its first half) and V_{u-1} (its
    // second half), so that one barrier covers a step's bytes (slot u = 0
    // holds K_0 alone, slot u = n V_{n-1} alone).
    static constexpr int STAGES = SLOTS_;
    static constexpr int BM = 128;                  // two query blocks
    static constexpr int BN = 128;                  // two key blocks
    static constexpr int NCH = D / 64;              // 64-column chunks per row
    static constexpr int Q_BYTES = NCH * BM * 128;
    static constexpr int KV_BYTES = NCH * BN * 128;  // one K or V tile
    static constexpr int SLOT_BYTES = 2 * KV_BYTES;
    static constexpr int NUM_BARS = 3 * STAGES + 6;
    static constexpr int SMEM_BYTES = 1024 + Q_BYTES + STAGES * SLOT_BYTES + NUM_BARS * 8 + 16;
    static constexpr int TMEM_S = 0;           // S buffers at [0, BN) and [BN, 2 BN)
    static constexpr int TMEM_O = 2 * BN;      // O at [2 BN, 2 BN + D)
    static constexpr int TMEM_P = 2 * BN + D;  // P buffers (bf16 pairs) at [TMEM_P, + BN / 2) and [+ BN / 2, + BN)
    static constexpr int TMEM_COLS = 512;
    static_assert(D % 64 == 0 && 3 * BN + D <= TMEM_COLS, "tile shape");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(SMEM_BYTES > 232448 / 2, "one CTA per SM: the TMEM allocation is 512 columns");
};

constexpr float kVsaLn2 = 0.6931471805599453f;
constexpr float kVsaRescale = 8.0f;  // log2 units: tolerate P up to 2^8 before rescaling O

// Token count of the key block of list entry e (clamped to [0, 64]; 0 for no block).
__device__ __forceinline__ int entry_rows_of(int e, int nb) {
    const int blk = e >> 9;
    if (e < 0 || blk >= nb) return 0;
    const int s = (e >> 2) & 127;
    return s < kVsaBlock ? s : kVsaBlock;
}

// Visible keys of a 64-row key block for the rows of query block qb (0 or 1)
// of the tile: its token count if that query block keeps it, else 0.
__device__ __forceinline__ int entry_keys(int e, int qb, int nb) {
    if (e < 0) return 0;
    const int blk = e >> 9;
    if (blk >= nb || !((e >> qb) & 1)) return 0;
    const int s = (e >> 2) & 127;
    return s < kVsaBlock ? s : kVsaBlock;
}

template <class C>
__global__ void __launch_bounds__(224, 1)
    vsa_fwd_sm103a(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const VsaFwdParams p) {
    constexpr int D = C::D, BN = C::BN, STAGES = C::STAGES, BM = C::BM, NCH = C::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + C::Q_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::Q_BYTES + STAGES * C::SLOT_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t b_q_full = smem_u32(&bars[0]);
    auto b_kv_full = [&](int s) { return smem_u32(&bars[1 + s]); };
    auto b_kv_empty = [&](int s) { return smem_u32(&bars[1 + STAGES + s]); };
    auto b_s_full = [&](int b) { return smem_u32(&bars[1 + 2 * STAGES + b]); };
    const uint32_t b_p_full = smem_u32(&bars[3 + 2 * STAGES]);
    const uint32_t b_pv_done = smem_u32(&bars[4 + 2 * STAGES]);
    const uint32_t b_drain = smem_u32(&bars[5 + 2 * STAGES]);
    // stage s's load has landed and, for a V tile, its padding rows are zeroed
    auto b_v_ready = [&](int s) { return smem_u32(&bars[6 + 2 * STAGES + s]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ------------------------------------------------------------ tile coordinates
    // The dense tiles (prefix query blocks keep every key block) of every head
    // start first, heads fastest; then each head's sparse tiles, tiles fastest,
    // so that the CTAs resident at one time read the K/V of one or two heads,
    // which stay in L2.
    int h, t;
    {
        const int dense = p.Hq * p.g.td, per = p.g.nt - p.g.td;
        const int L = blockIdx.x;
        if (L < dense) {
            h = L % p.Hq;
            t = L / p.Hq;
        } else {
            h = (L - dense) / per;
            t = p.g.td + (L - dense) % per;
        }
    }
    const int kvh = h / p.group;
    const int nb = p.g.nb;
    const int cap = p.g.capacity(t);
    const int32_t* list = p.kv_list + static_cast<long long>(h) * p.g.per_head() + p.g.offset(t);
    int n = p.kv_num[static_cast<long long>(h) * p.g.nt + t];
    if (n < 0 || n > cap) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, kDevBadIndex);
        n = n < 0 ? 0 : cap;
    }
    const int n_kv = (n + 1) >> 1;  // KV tile j = entries 2 j and 2 j + 1
    if (status_has_timeout(p.status, kDevTimeout)) return;

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(b_kv_full(s), 1);
            mbar_init(b_kv_empty(s), 1);
            mbar_init(b_v_ready(s), 1);
        }
        mbar_init(b_s_full(0), 1);
        mbar_init(b_s_full(1), 1);
        mbar_init(b_p_full, 128);
        mbar_init(b_pv_done, 1);
        mbar_init(b_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(b_q_full, C::Q_BYTES);
            for (int c = 0; c < NCH; ++c) tma_load_3d(sQ + c * BM * 128, &tmQ, b_q_full, c * 64, h, t * BM);
            // Slot load u: K_u (entries 2u, 2u + 1) in its first half for u < n,
            // V_{u-1} (the previous K tile's blocks) in its second for u >= 1.
            // A missing second entry repeats the first block (masked for every
            // row); a bad entry is flagged and block 0 read instead.
            int issued = 0;
            int vb0 = 0, vb1 = 0;  // blocks of the previous K tile
            int ne0 = 0, ne1 = -1;  // entries of the next K tile, read one load ahead
            if (n_kv > 0) {
                ne0 = list[0];
                ne1 = n > 1 ? list[1] : -1;
            }
            for (int u = 0; ok && n_kv > 0 && u <= n_kv; ++u) {
                const bool hk = u < n_kv, hv = u >= 1;
                int b0 = 0, b1 = 0;
                if (hk) {
                    const int e0 = ne0, e1 = ne1;
                    if (u + 1 < n_kv) {
                        ne0 = list[2 * u + 2];
                        ne1 = 2 * u + 3 < n ? list[2 * u + 3] : -1;
                    }
                    b0 = e0 >> 9;
                    b1 = e1 < 0 ? b0 : (e1 >> 9);
                    if (b0 < 0 || b0 >= nb || b1 < 0 || b1 >= nb) {
                        if (p.status) atomicOr(p.status, kDevBadIndex);
                        b0 = (b0 < 0 || b0 >= nb) ? 0 : b0;
                        b1 = (b1 < 0 || b1 >= nb) ? 0 : b1;
                    }
                }
                const int s = u % STAGES, w = u / STAGES;
                if (w > 0 && !mbar_wait(b_kv_empty(s), (w - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = sKV + s * C::SLOT_BYTES;
                mbar_arrive_expect_tx(b_kv_full(s), (hk ? C::KV_BYTES : 0) + (hv ? C::KV_BYTES : 0));
                for (int c = 0; c < NCH; ++c) {
                    if (hk) {
                        tma_load_3d(dst + c * BN * 128, &tmK, b_kv_full(s), c * 64, kvh, b0 * kVsaBlock);
                        tma_load_3d(dst + c * BN * 128 + kVsaBlock * 128, &tmK, b_kv_full(s), c * 64, kvh,
                                    b1 * kVsaBlock);
                    }
                    if (hv) {
                        tma_load_3d(dst + C::KV_BYTES + c * BN * 128, &tmV, b_kv_full(s), c * 64, kvh, vb0 * kVsaBlock);
                        tma_load_3d(dst + C::KV_BYTES + c * BN * 128 + kVsaBlock * 128, &tmV, b_kv_full(s), c * 64,
                                    kvh, vb1 * kVsaBlock);
                    }
                }
                vb0 = b0;
                vb1 = b1;
                ++issued;
            }
            if (!ok || *abort_flag) {
                // Let every copy this thread started land before the CTA retires.
                mbar_wait_drain(b_q_full, 0);
                for (int u_ = (issued > STAGES ? issued - STAGES : 0); u_ < issued; ++u_)
                    mbar_wait_drain(b_kv_full(u_ % STAGES), (u_ / STAGES) & 1);
            }
        }
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        // The whole warp walks the schedule; one elected lane issues.
        constexpr uint32_t kIdS = idesc_bf16_f32(BM, BN, false, false);
        constexpr uint32_t kIdO = idesc_bf16_f32(BM, D, false, true);
        const bool leader = elect_one();
        const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
        const uint64_t dK = sdesc_sw128(sKV, 16, 1024);
        const uint64_t dV = sdesc_sw128(sKV + C::KV_BYTES, BN * 128, 1024);
        auto wait_all = [&](uint32_t bar, uint32_t ph) {
            return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort_flag));
        };
        auto issue_s = [&](int j, int s) {  // S_j from the K half of slot s
            if (leader) {
                const uint32_t dS = tmem + C::TMEM_S + (j & 1) * BN;
                const uint64_t b0 = dK + static_cast<uint64_t>(s * (C::SLOT_BYTES >> 4));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * BM * 128 + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(dS, dQ + oa, b0 + ob, kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(b_s_full(j & 1));
            }
            __syncwarp();
        };
        ok = wait_all(b_q_full, 0);
        if (ok && n_kv > 0 && (ok = wait_all(b_kv_full(0), 0))) {  // slot load 0: K_0 alone
            tc_fence_after();
            issue_s(0, 0);
            if (leader) mma_commit(b_kv_empty(0));
            __syncwarp();
        }
        for (int j = 0; ok && j < n_kv; ++j) {
            // slot load j + 1: K_{j+1} (but for the last step) and V_j
            const int s = (j + 1) % STAGES;
            const uint32_t ph = static_cast<uint32_t>((j + 1) / STAGES) & 1u;
            if (!(ok = wait_all(b_kv_full(s), ph))) break;
            tc_fence_after();
            if (j + 1 < n_kv) issue_s(j + 1, s);
            if (!(ok = wait_all(b_p_full, j & 1))) break;
            if (!(ok = wait_all(b_v_ready(s), ph))) break;  // V_j's padding rows zeroed
            tc_fence_after();
            if (leader) {
                // O += P_j V_j, P_j (bf16 pairs) read from its TMEM buffer
                const uint64_t b0 = dV + static_cast<uint64_t>(s * (C::SLOT_BYTES >> 4));
                const uint32_t a = tmem + C::TMEM_P + (j & 1) * (BN / 2);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16_ts(tmem + C::TMEM_O, a + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdO,
                                (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(b_pv_done);
                mma_commit(b_kv_empty(s));
            }
            __syncwarp();
        }
        if (leader) mma_commit(b_drain);  // all of the above finishes before TMEM is released
        __syncwarp();
        mbar_wait_drain(b_drain, 0);
    } else if (warp == 6) {
        // ----------------------------------------------------------- V padding
        // Rows of a V tile past each key block's token count are padding,
        // which may hold anything, NaN included; P is 0 there but 0 * NaN is
        // not.  This warp follows the ring in load order: once a slot load
        // has landed it zeroes the padding rows of its V tile, then passes
        // the slot on (b_v_ready), which the MMA warp waits for before P V.
        // It passes slot load 0 (K_0 alone) on too, after it lands, so that
        // no slot's b_v_ready runs a phase ahead of its loads.
        for (int u = 0; ok && n_kv > 0 && u <= n_kv; ++u) {
            const int s = u % STAGES;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_kv_full(s), (u / STAGES) & 1, abort_flag)))) break;
            if (u >= 1) {  // V_{u-1} in the slot's second half
                const int jv = u - 1;
                const int ea = list[2 * jv], eb = 2 * jv + 1 < n ? list[2 * jv + 1] : -1;
                const int za = entry_rows_of(ea, nb), zb = eb < 0 ? 0 : entry_rows_of(eb, nb);
                if (za < kVsaBlock || zb < kVsaBlock) {
                    const uint32_t vb = sKV + s * C::SLOT_BYTES + C::KV_BYTES;
                    const int na = kVsaBlock - za, nz = na + kVsaBlock - zb;
                    for (int idx = lane; idx < nz * NCH * 8; idx += 32) {
                        const int uu = idx & 7, rc = idx >> 3, c = rc % NCH, k = rc / NCH;
                        const int rr = k < na ? za + k : kVsaBlock + zb + (k - na);
                        st_shared_v4(vb + c * BN * 128 + rr * 128 + uu * 16, 0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(b_v_ready(s));
        }
    } else {
        // ------------------------------------------------------------- softmax
        const int r = threadIdx.x;  // row within the tile == TMEM lane
        const int qb = r >> 6;      // query block of the row within the pair (warp-uniform)
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float c2 = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        int e0 = n > 0 ? list[0] : 0, e1 = n > 1 ? list[1] : -1;
        for (int j = 0; j < n_kv; ++j) {
            int f0 = 0, f1 = -1;
            if (j + 1 < n_kv) {
                f0 = list[2 * j + 2];
                f1 = 2 * j + 3 < n ? list[2 * j + 3] : -1;
            }
            const int la = entry_keys(e0, qb, nb), lb = entry_keys(e1, qb, nb);
            e0 = f0;
            e1 = f1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_s_full(j & 1), (j >> 1) & 1, abort_flag)))) break;
            tc_fence_after();
            const uint32_t tS = tl + C::TMEM_S + (j & 1) * BN;
            uint32_t pk[BN / 2];
            bool warp_need = false;
            float alpha = 1.f;
            if (la > 0 || lb > 0) {
                uint32_t sr[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c)
                    tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
                tmem_wait_ld();
                if (la < kVsaBlock || lb < kVsaBlock) {
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c < kVsaBlock ? c >= la : c - kVsaBlock >= lb) sr[c] = __float_as_uint(-INFINITY);
                }
                float mxp[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) mxp[i] = __uint_as_float(sr[i]);
#pragma unroll
                for (int c = 4; c < BN; c += 2)
                    mxp[(c >> 1) & 3] = fmax3(mxp[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                const float mx = fmaxf(fmax3(mxp[0], mxp[1], mxp[2]), mxp[3]);
                const float m_new = fmaxf(m, mx * c2);
                warp_need = __any_sync(0xffffffffu, m_new > m + kVsaRescale);
                if (warp_need && m_new > m) {
                    alpha = ex2(m - m_new);
                    m = m_new;
                }
                l *= alpha;
                const float msub = (m == -INFINITY) ? 0.f : m;
                const float2 c2x2 = make_float2(c2, c2), negm = make_float2(-msub, -msub);
                float2 rsp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < BN; c += 2) {
                    const float2 x =
                        __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2x2, negm);
                    const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                    rsp[(c >> 1) & 3] = __fadd2_rn(rsp[(c >> 1) & 3], pp);
                    pk[c >> 1] = pack_bf16x2(pp.x, pp.y);
                }
                const float2 rr = __fadd2_rn(__fadd2_rn(rsp[0], rsp[1]), __fadd2_rn(rsp[2], rsp[3]));
                l += rr.x + rr.y;
            } else {  // this query block keeps neither key block: P = 0, m and l unchanged
#pragma unroll
                for (int c = 0; c < BN / 2; ++c) pk[c] = 0u;
            }
            // PV_{j-1} is complete before P_j is released (and before O is
            // rescaled): S_j was issued after PV_{j-2} only, so here PV_{j-2}
            // is complete and PV_j not yet issued, and pv_done has completed
            // j - 1 or j phases; a wait on the parity of phase j - 1 is exact
            // whichever it is.  P_j replaces P_{j-2} in buffer j & 1.  (Waiting
            // only when O is rescaled, as the prefill kernels do, measured the
            // same speed here and gave wrong rows at D = 64.)
            if (j > 0) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_pv_done, (j - 1) & 1, abort_flag)))) break;
                tc_fence_after();
                if (warp_need) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tl + C::TMEM_O + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tl + C::TMEM_O + c * 32, o);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_st16(tl + C::TMEM_P + (j & 1) * (BN / 2) + c * 16, &pk[c * 16]);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_p_full);
        }
        ok = __all_sync(0xffffffffu, ok);
        if (ok && n_kv > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_pv_done, (n_kv - 1) & 1, abort_flag));
            tc_fence_after();
        }
        // ------------------------------------------------------------ epilogue
        // Row r of the tile goes to row out_index[t * 128 + r] of out (the
        // token's place in the sequence), or nowhere when that is negative.
        const long long R = static_cast<long long>(t) * BM + r;
        long long orow = p.out_index ? static_cast<long long>(p.out_index[R]) : R;
        if (orow >= p.out_rows) {
            if (p.status) atomicOr(p.status, kDevBadIndex);
            orow = -1;
        }
        const bool row_valid = ok && orow >= 0;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const long long obase = (orow * p.Hq + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (n_kv > 0 && ok) {
                tmem_ld32(tl + C::TMEM_O + c * 32, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (row_valid) {
                if (p.out_f32) {
                    float* dst = reinterpret_cast<float*>(p.out) + obase + c * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        st_global_v4(dst + e, __float_as_uint(__uint_as_float(o[e]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 1]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 2]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 3]) * inv_l));
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + obase + c * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        st_global_v4(dst + e,
                                     pack_bf16x2(__uint_as_float(o[e]) * inv_l, __uint_as_float(o[e + 1]) * inv_l),
                                     pack_bf16x2(__uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l),
                                     pack_bf16x2(__uint_as_float(o[e + 4]) * inv_l, __uint_as_float(o[e + 5]) * inv_l),
                                     pack_bf16x2(__uint_as_float(o[e + 6]) * inv_l, __uint_as_float(o[e + 7]) * inv_l));
                }
            }
        }
        if (row_valid && p.lse)
            p.lse[static_cast<long long>(h) * p.out_rows + orow] = l > 0.f ? (m + __log2f(l)) * kVsaLn2 : -INFINITY;
    }

    // --------------------------------------------------------------- teardown
    if (!ok) {
        *abort_flag = 1;
        if (p.status) atomicOr(p.status, kDevTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

using VsaCfg64 = VsaCfg<64, 6>;
using VsaCfg128 = VsaCfg<128, 3>;

// ------------------------------------------------------------------ launchers
static int grid_for(long long units, int per_cta, int num_sms, int ctas_per_sm) {
    long long g = (units + per_cta - 1) / per_cta;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * ctas_per_sm;
    return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

cudaError_t launch_gather_rows(const void* src, long long src_rows, const int32_t* index, long long dst_rows,
                               int row_bytes, void* dst, uint32_t* status, int num_sms, cudaStream_t st) {
    gather_rows_sm103a<<<grid_for(dst_rows, 8, num_sms, 8), 256, 0, st>>>(
        static_cast<const uint4*>(src), src_rows, index, dst_rows, row_bytes / 16, static_cast<uint4*>(dst), status);
    return cudaGetLastError();
}

cudaError_t launch_vsa_pool(const void* x, const int32_t* sizes, int nb, int H, int D, float* pooled,
                            uint32_t* status, int num_sms, cudaStream_t st) {
    const long long units = static_cast<long long>(nb) * H * (D / 8);
    vsa_pool_sm103a<<<grid_for(units, 256, num_sms, 8), 256, 0, st>>>(static_cast<const uint4*>(x), sizes, nb, H, D,
                                                                    pooled, status);
    return cudaGetLastError();
}

int vsa_map_smem_bytes(int nb, int D, int qb) {
    const long long words = (nb + 31) / 32;
    const long long b = 4LL * (static_cast<long long>(kMapQB) * D + kMapKeys * kMapKS + static_cast<long long>(qb) * nb +
                               qb * words) +
                        4LL * kMapWarps * 256;
    return b > 232448 ? -1 : static_cast<int>(b);
}

cudaError_t launch_vsa_block_map(const float* pq, const float* pk, const int32_t* sizes, const VsaGeom& g, int Hq,
                                 int group, int D, float scale, int32_t* kv_list, int32_t* kv_num, uint32_t* status,
                                 cudaStream_t st) {
    int qb = kMapQB;
    while (qb > 2 && vsa_map_smem_bytes(g.nb, D, qb) < 0) qb >>= 1;
    const int bytes = vsa_map_smem_bytes(g.nb, D, qb);
    if (bytes < 0) return cudaErrorInvalidValue;
    // Per device, the kernel's dynamic shared-memory limit only ever rises
    // (to the largest size asked for so far), so a launch made after another
    // thread's smaller request still finds its own size allowed.
    static int high[64];
    static std::mutex mu;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || bytes > high[dev]) {
            e = cudaFuncSetAttribute(vsa_block_map_sm103a, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) high[dev] = bytes;
        }
    }
    VsaMapParams p{pq, pk, sizes, kv_list, kv_num, status, g, group, D, qb, scale};
    dim3 grid((g.nb + qb - 1) / qb, Hq);
    vsa_block_map_sm103a<<<grid, kMapWarps * 32, bytes, st>>>(p);
    return cudaGetLastError();
}

template <class C>
static cudaError_t launch_vsa_cfg(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const VsaFwdParams& p, cudaStream_t st) {
    static bool done[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !done[dev]) {
            e = cudaFuncSetAttribute(vsa_fwd_sm103a<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) done[dev] = true;
        }
    }
    const long long ctas = static_cast<long long>(p.Hq) * p.g.nt;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    vsa_fwd_sm103a<C><<<static_cast<unsigned>(ctas), 224, C::SMEM_BYTES, st>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

cudaError_t launch_vsa_fwd(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const VsaFwdParams& p, cudaStream_t st) {
    switch (D) {
        case 64: return launch_vsa_cfg<VsaCfg64>(tmQ, tmK, tmV, p, st);
        case 128: return launch_vsa_cfg<VsaCfg128>(tmQ, tmK, tmV, p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbattn
