// decode.cu -- paged-KV decode (one query token per sequence) for sm_103a.
//
// Operation: vllm-ascend attention_v1.py, AscendAttentionBackendImpl.
// forward_paged_attention -- each sequence's query attends its whole context,
// read from the cache (2, num_blocks, 128, Hkv, D) through block_table and
// seq_lens (AscendAttentionBackend.get_kv_cache_shape; token t of sequence s
// is slot t % 128 of block block_table[s, t / 128], the AscendMetadata
// slot_mapping rule).
//
// The path is HBM-bound, so it runs on the CUDA cores.  Design:
//   * work item = (sequence, split of up to `blocks_per_split` cache blocks,
//     KV head [, query-head subgroup]); paged_schedule (one CTA) lists the
//     non-empty (sequence, split) pairs longest first, and a persistent grid
//     of one CTA per SM claims items from a global counter, KV heads varying
//     fastest so that the CTAs working at one moment read neighbouring
//     256-byte head rows of the same cache rows;
//   * the K and V of one slice (a whole 128-token block, or 64 tokens at
//     D >= 192) arrive by TMA as one box per 64 columns into a ring of
//     shared-memory slots (large boxes: the TMA issue cost per box, not the
//     bytes, limits small-box streaming);
//   * all 8 warps consume every slot, each a fixed run of its tokens, so
//     every mbarrier phase is awaited in order; there is no producer warp:
//     the last warp to release a slot (a shared-memory counter) refills it
//     with the next slice, claiming a new item when the current one is
//     exhausted, and records the slice's item in the slot's header;
//   * inside a warp a group of LPG lanes owns one token at a time, each lane
//     E = D / LPG columns, with the GQA group's query rows for those columns
//     in registers: q.k is a packed-fp32 (fma.rn.f32x2) dot product plus a
//     log2(LPG)-level shuffle reduction, o += p.v reuses the same columns, so
//     each K and V byte is read from shared memory once for all HG heads;
//   * each warp keeps its own online softmax; at the end of an item the
//     groups and warps merge (m, l, o) by the log-sum-exp rule and write the
//     item's partial (o / l, lse); paged_combine merges the splits:
//     lse = ln sum_i exp(lse_i), o = sum_i exp(lse_i - lse) o_i.
// Tokens at or past seq_len are never used, neither in q.k nor in p.v, so
// whatever the unused cache slots hold cannot reach the result.
#include <math.h>

#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {

constexpr int kBlk = 128;  // tokens per cache block
constexpr int kWarps = 8;  // all of them consume every slot
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D_, int HG_>
struct PagedCfg {
    static constexpr int D = D_;
    static constexpr int HG = HG_;                       // query heads per CTA (divides the GQA group)
    static constexpr int SLICE = D <= 128 ? 128 : 64;    // tokens per slot
    // columns per lane: at most 64 / HG (q and o stay in registers), and small
    // enough that every warp owns at least one token step of a slice
    static constexpr int E0 = (D % 96 == 0) ? 48 / HG : 64 / HG;
    static constexpr int EMAX = D * SLICE / (32 * kWarps);
    static constexpr int E = E0 < EMAX ? E0 : EMAX;
    static constexpr int LPG = D / E;                    // lanes per token group
    static constexpr int TPW = 32 / LPG;                 // tokens a warp handles per step
    static constexpr int NSTEP = SLICE / TPW;            // steps per slot
    static constexpr int WSTEP = NSTEP / kWarps;         // steps per warp per slot
    static constexpr int SUBS = WSTEP < 32 / HG ? WSTEP : 32 / HG;  // steps per softmax sub-chunk
    static constexpr int NCH = (D + 63) / 64;
    static constexpr int HALF_BYTES = NCH * SLICE * 128;  // K (or V) of one slice
    static constexpr int SLOT_BYTES = 2 * HALF_BYTES;
    static constexpr int MERGE_BYTES = kWarps * HG * (D + 2) * 4;
    static constexpr int STAGES_RAW = (230400 - MERGE_BYTES) / SLOT_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    // vector width of one shared-memory load, in bf16 elements
    static constexpr int U = (E % 8 == 0) ? 8 : ((E % 4 == 0) ? 4 : 2);
    // period (in steps) of a lane's swizzle pattern: rows advance by TPW per step, the swizzle by row % 8
    static constexpr int P = TPW >= 8 ? 1 : 8 / TPW;
    // shared memory: slots | merge scratch [warps][HG][D + 2] f32 | counters | slot headers | uses | cursor | bars
    static constexpr int OFF_MERGE = STAGES * SLOT_BYTES;
    static constexpr int OFF_CNT = OFF_MERGE + MERGE_BYTES;
    static constexpr int OFF_INFO = OFF_CNT + STAGES * 4;
    static constexpr int OFF_USE = OFF_INFO + STAGES * 32;
    static constexpr int OFF_CUR = OFF_USE + STAGES * 4;
    static constexpr int OFF_BAR = (OFF_CUR + 32 + 7) & ~7;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + STAGES * 8;
    static_assert(LPG * E == D && 32 % LPG == 0 && SLICE % TPW == 0 && NSTEP % kWarps == 0 && WSTEP % SUBS == 0,
                  "lane map");
    static_assert(STAGES >= 2 && SMEM_BYTES <= 232448, "shared memory budget");
    static_assert((WSTEP * TPW) % 8 == 0, "each warp's rows start 8-aligned");
};

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Header of one slot, written by the thread that fills it.
struct SlotInfo {
    int item;  // -1: end of this CTA's work
    int s, h0, kvh, sp, tok, tok1;
    int bad;   // the block id was outside [0, num_blocks): no data, tokens skipped
};

// The refill cursor: the next slice to load.  Only one thread at a time
// touches it (refills happen in slice order, handed from one releasing warp
// to the next through the slot counters' acquire/release atomics).
struct Cursor {
    int item, s, h0, kvh, sp, tok, tok1;
};

__device__ __forceinline__ void claim_item(const PagedParams& p, int n_hgroups, int total, Cursor& cu) {
    const int k = atomicAdd(p.sched, 1);
    if (k >= total) {
        cu.item = -1;
        return;
    }
    const int4 pr = p.pairs[k / n_hgroups];
    const int hg = k % n_hgroups;
    const int per_kv = p.group / p.heads_per_cta;
    cu.item = k;
    cu.s = pr.x;
    cu.sp = pr.y;
    cu.tok = pr.z;
    cu.tok1 = pr.w;
    cu.kvh = hg / per_kv;
    cu.h0 = cu.kvh * p.group + (hg % per_kv) * p.heads_per_cta;
}

// This lane's E columns of one token row as E/2 packed words: `base[u]` is
// the shared address of the lane's u-th vector for row offset 0 (swizzle
// already applied), `imm` a compile-time row offset that keeps the swizzle
// phase (a multiple of 8 rows, plus the K->V distance).
template <class C>
__device__ __forceinline__ void lds_cols(const uint32_t (&base)[C::E / C::U], uint32_t imm, uint32_t (&w)[C::E / 2]) {
#pragma unroll
    for (int u = 0; u < C::E / C::U; ++u) {
        const uint32_t addr = base[u] + imm;
        if constexpr (C::U == 8) {
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[u * 4]), "=r"(w[u * 4 + 1]), "=r"(w[u * 4 + 2]), "=r"(w[u * 4 + 3])
                         : "r"(addr));
        } else if constexpr (C::U == 4) {
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(w[u * 2]), "=r"(w[u * 2 + 1]) : "r"(addr));
        } else {
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[u]) : "r"(addr));
        }
    }
}

// Fill `slot` with the cursor's slice (one thread) and advance the cursor.
// A block id outside [0, num_blocks) is reported; the slot is then marked bad
// and its barrier completed without data.  An exhausted cursor writes the
// end marker.
template <class C>
__device__ __forceinline__ void fill_slot(const CUtensorMap* tm, const PagedParams& p, uint32_t sSlots, uint32_t bar,
                                          volatile SlotInfo* info, volatile int* suse, int slot, int use,
                                          Cursor& cu, int n_hgroups, int total) {
    volatile SlotInfo& si = info[slot];
    suse[slot] = use;
    si.item = cu.item;
    if (cu.item < 0) {
        mbar_arrive(bar);
        return;
    }
    si.s = cu.s;
    si.h0 = cu.h0;
    si.kvh = cu.kvh;
    si.sp = cu.sp;
    si.tok = cu.tok;
    si.tok1 = cu.tok1;
    const int blk = p.block_table[static_cast<long long>(cu.s) * p.max_blocks_per_seq + cu.tok / kBlk];
    const bool valid = blk >= 0 && blk < p.num_blocks;
    si.bad = valid ? 0 : 1;
    if (valid) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, C::SLOT_BYTES);
        const int row = blk * kBlk + (cu.tok & (kBlk - 1));
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
            for (int ch = 0; ch < C::NCH; ++ch)
                tma_load_3d(sSlots + slot * C::SLOT_BYTES + kv * C::HALF_BYTES + ch * C::SLICE * 128, tm, bar,
                            ch * 64, cu.kvh, row + kv * p.num_blocks * kBlk);
    } else {
        if (p.status) atomicOr(p.status, kDevBadIndex);
        mbar_arrive(bar);
    }
    cu.tok += C::SLICE;
    if (cu.tok >= cu.tok1) claim_item(p, n_hgroups, total, cu);
}

template <class C>
__global__ void __launch_bounds__(32 * kWarps, 1)
    paged_decode_sm103a(const __grid_constant__ CUtensorMap tmKV, const PagedParams p) {
    constexpr int D = C::D, HG = C::HG, E = C::E, LPG = C::LPG, TPW = C::TPW, STAGES = C::STAGES;
    constexpr int SLICE = C::SLICE, WSTEP = C::WSTEP, SUBS = C::SUBS, P = C::P, NU = C::E / C::U;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sSlots = smem_u32(smem);
    float* smerge = reinterpret_cast<float*>(smem + C::OFF_MERGE);  // [warp][HG][D + 2]: o..., m, l
    int* scnt = reinterpret_cast<int*>(smem + C::OFF_CNT);          // releases per slot, monotonic
    volatile SlotInfo* sinfo = reinterpret_cast<volatile SlotInfo*>(smem + C::OFF_INFO);
    volatile int* suse = reinterpret_cast<volatile int*>(smem + C::OFF_USE);  // last use filled per slot
    Cursor* scur = reinterpret_cast<Cursor*>(smem + C::OFF_CUR);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    auto b_full = [&](int s) { return smem_u32(&bars[s]); };
    __shared__ int abort_flag_storage;
    volatile int* abort_flag = &abort_flag_storage;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_hgroups = p.Hkv * (p.group / p.heads_per_cta);
    if (status_has_timeout(p.status, kDevTimeout)) return;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(b_full(s), 1);
            scnt[s] = 0;
            suse[s] = -1;
        }
        abort_flag_storage = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmKV);
    }
    // Launched behind paged_schedule, which may still run: its list and
    // counters are read only past this point.
    grid_dependency_wait();
    grid_launch_dependents();  // paged_combine may queue up (it waits for this grid)
    const int total = p.sched[1] * n_hgroups;  // items in this launch
    __syncthreads();
    if (threadIdx.x == 0) {  // prologue: the first STAGES slices
        Cursor cu;
        claim_item(p, n_hgroups, total, cu);
        for (int s = 0; s < STAGES; ++s) fill_slot<C>(&tmKV, p, sSlots, b_full(s), sinfo, suse, s, 0, cu, n_hgroups, total);
        *scur = cu;
    }
    bool ok = true;
    const float c2 = p.scale_log2;
    const int grp = lane / LPG;       // token group within the warp
    const int e0 = (lane % LPG) * E;  // this lane's first column
    // byte offset of this lane's u-th load of row (j * TPW + grp), j < P
    uint32_t loff[P][NU];
#pragma unroll
    for (int j = 0; j < P; ++j) {
        const int row = j * TPW + grp;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int e = e0 + u * C::U;
            loff[j][u] = (e >> 6) * (SLICE * 128) + row * 128 + ((((e & 63) >> 3) ^ (row & 7)) << 4) + (e & 7) * 2;
        }
    }
    int cur_item = -1, cur_s = 0, cur_h0 = 0, cur_sp = 0;
    float2 q[HG][E / 2];
    float m[HG], l[HG];
    float2 o[HG][E / 2];

    // Merge the token groups and warps of the finished item, write its partial.
    auto finish_item = [&]() {
#pragma unroll
        for (int off = LPG; off < 32; off <<= 1) {
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
                const float mt = fmaxf(m[h], mo);
                const float a = (m[h] == -INFINITY) ? 0.f : ex2(m[h] - mt);
                const float b = (mo == -INFINITY) ? 0.f : ex2(mo - mt);
                l[h] = l[h] * a + lo * b;
#pragma unroll
                for (int x = 0; x < E / 2; ++x) {
                    const float ox = __shfl_xor_sync(0xffffffffu, o[h][x].x, off);
                    const float oy = __shfl_xor_sync(0xffffffffu, o[h][x].y, off);
                    o[h][x] = make_float2(o[h][x].x * a + ox * b, o[h][x].y * a + oy * b);
                }
                m[h] = mt;
            }
        }
        if (grp == 0) {
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float* dst = smerge + (warp * HG + h) * (D + 2);
#pragma unroll
                for (int x = 0; x < E / 2; ++x) {
                    dst[e0 + 2 * x] = o[h][x].x;
                    dst[e0 + 2 * x + 1] = o[h][x].y;
                }
                if (lane == 0) {
                    dst[D] = m[h];
                    dst[D + 1] = l[h];
                }
            }
        }
        __syncthreads();
        for (int x = threadIdx.x; x < HG * D; x += 32 * kWarps) {
            const int h = x / D, d = x % D;
            float mt = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) mt = fmaxf(mt, smerge[(w * HG + h) * (D + 2) + D]);
            float lt = 0.f, ot = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* src = smerge + (w * HG + h) * (D + 2);
                const float a = (src[D] == -INFINITY) ? 0.f : ex2(src[D] - mt);
                lt = fmaf(src[D + 1], a, lt);
                ot = fmaf(src[d], a, ot);
            }
            const long long row = (static_cast<long long>(cur_s) * p.Hq + cur_h0 + h) * p.max_splits + cur_sp;
            p.part_o[row * D + d] = lt > 0.f ? ot / lt : 0.f;
            if (d == 0) p.part_lse[row] = lt > 0.f ? (mt + __log2f(lt)) * kLn2f : -INFINITY;
        }
        __syncthreads();
    };

    for (int g = 0;; ++g) {
        const int slot = g % STAGES, use = g / STAGES;
        if (!mbar_wait(b_full(slot), use & 1, abort_flag)) {
            ok = false;
            *abort_flag = 1;
        }
        ok = __all_sync(0xffffffffu, ok);
        // every warp reads the same header, so every warp leaves at the same slice
        const int item = ok ? sinfo[slot].item : -1;
        if (item < 0) break;
        if (item != cur_item) {
            // The barriers of the kernel are those of finish_item.  A warp whose
            // wait succeeded after another warp gave up (data arriving just
            // after the give-up) reads the abort flag here, before any barrier,
            // and leaves too: no warp finishes an item another warp abandoned,
            // and no partial is written after a give-up (the status word
            // reports it), so every warp passes the same number of barriers.
            if (__any_sync(0xffffffffu, *abort_flag != 0)) {
                ok = false;
                break;
            }
            if (cur_item >= 0) finish_item();
            cur_item = item;
            cur_s = sinfo[slot].s;
            cur_h0 = sinfo[slot].h0;
            cur_sp = sinfo[slot].sp;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const uint16_t* qh = reinterpret_cast<const uint16_t*>(p.q) +
                                     (static_cast<long long>(cur_s) * p.Hq + cur_h0 + h) * D + e0;
#pragma unroll
                for (int x = 0; x < E / 2; ++x) {
                    const uint32_t qq = *reinterpret_cast<const uint32_t*>(qh + 2 * x);
                    q[h][x] = make_float2(bf_lo(qq), bf_hi(qq));
                }
                m[h] = -INFINITY;
                l[h] = 0.f;
#pragma unroll
                for (int x = 0; x < E / 2; ++x) o[h][x] = make_float2(0.f, 0.f);
            }
        }
        const int nvalid = sinfo[slot].bad ? 0 : min(SLICE, sinfo[slot].tok1 - sinfo[slot].tok);
        // this warp's K rows start 8-aligned, so every lane's swizzled offsets repeat with period P steps
        uint32_t kl[P][NU];
#pragma unroll
        for (int j = 0; j < P; ++j)
#pragma unroll
            for (int u = 0; u < NU; ++u) kl[j][u] = sSlots + slot * C::SLOT_BYTES + warp * (WSTEP * TPW * 128) + loff[j][u];
        auto process = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
            for (int sc = 0; sc < WSTEP / SUBS; ++sc) {
                // ---- scores of SUBS tokens of this group, HG heads
                float s[SUBS][HG];
#pragma unroll
                for (int st = 0; st < SUBS; ++st) {
                    const int stg = sc * SUBS + st;
                    const int t = (warp * WSTEP + stg) * TPW + grp;
                    const bool live = FULL || t < nvalid;  // group-uniform
                    float dot[HG];
                    if (live) {
                        uint32_t w[E / 2];
                        lds_cols<C>(kl[stg % P], (stg - stg % P) * TPW * 128, w);
                        float2 acc[HG];
#pragma unroll
                        for (int h = 0; h < HG; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int x = 0; x < E / 2; ++x) {
                            const float2 kk = make_float2(bf_lo(w[x]), bf_hi(w[x]));
#pragma unroll
                            for (int h = 0; h < HG; ++h) acc[h] = __ffma2_rn(q[h][x], kk, acc[h]);
                        }
#pragma unroll
                        for (int h = 0; h < HG; ++h) dot[h] = acc[h].x + acc[h].y;
                    } else {
#pragma unroll
                        for (int h = 0; h < HG; ++h) dot[h] = 0.f;
                    }
#pragma unroll
                    for (int off = 1; off < LPG; off <<= 1)
#pragma unroll
                        for (int h = 0; h < HG; ++h) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], off);
#pragma unroll
                    for (int h = 0; h < HG; ++h) s[st][h] = live ? dot[h] * c2 : -INFINITY;
                }
                // ---- online softmax for this group (identical in its LPG lanes)
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    float cm = s[0][h];
#pragma unroll
                    for (int st = 1; st < SUBS; ++st) cm = fmaxf(cm, s[st][h]);
                    if (cm > m[h] + 8.0f) {  // rescale only when the max grows by more than 2^8
                        const float a = ex2(m[h] - cm);
                        const float2 a2 = make_float2(a, a);
                        l[h] *= a;
#pragma unroll
                        for (int x = 0; x < E / 2; ++x) o[h][x] = __fmul2_rn(o[h][x], a2);
                        m[h] = cm;
                    }
                    const float ms = (m[h] == -INFINITY) ? 0.f : m[h];
#pragma unroll
                    for (int st = 0; st < SUBS; ++st) {
                        s[st][h] = ex2(s[st][h] - ms);
                        l[h] += s[st][h];
                    }
                }
                // ---- o += p v over the same columns
#pragma unroll
                for (int st = 0; st < SUBS; ++st) {
                    const int stg = sc * SUBS + st;
                    const int t = (warp * WSTEP + stg) * TPW + grp;
                    if (FULL || t < nvalid) {
                        uint32_t w[E / 2];
                        lds_cols<C>(kl[stg % P], (stg - stg % P) * TPW * 128 + C::HALF_BYTES, w);
#pragma unroll
                        for (int x = 0; x < E / 2; ++x) {
                            const float2 vv = make_float2(bf_lo(w[x]), bf_hi(w[x]));
#pragma unroll
                            for (int h = 0; h < HG; ++h)
                                o[h][x] = __ffma2_rn(make_float2(s[st][h], s[st][h]), vv, o[h][x]);
                        }
                    }
                }
            }
        };
        if (nvalid == SLICE)
            process(std::true_type{});
        else
            process(std::false_type{});
        // ---- release the slot; the last warp out refills it with the next slice
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();  // this warp's reads of the slot happen before its release
            const int prev = atomicAdd(scnt + slot, 1);
            __threadfence_block();
            if (prev == use * kWarps + kWarps - 1 && !*abort_flag) {
                Cursor cu = *scur;
                fill_slot<C>(&tmKV, p, sSlots, b_full(slot), sinfo, suse, slot, use + 1, cu, n_hgroups, total);
                *scur = cu;
            }
        }
        __syncwarp();
    }
    if (cur_item >= 0 && ok) finish_item();  // after a give-up no partial is written (the status reports it)
    if (!ok) {
        *abort_flag = 1;
        if (p.status) atomicOr(p.status, kDevTimeout);
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {  // let copies still in flight land (bounded) before exit
        for (int s = 0; s < STAGES; ++s)
            if (suse[s] >= 0) mbar_wait_drain(b_full(s), suse[s] & 1);
    }
}

// One CTA: the non-empty (sequence, split) pairs, longest first (a counting
// sort on the split's block count, so the short last splits of the
// sequences come at the end), and the work counter reset to 0.  Reports
// seq_lens outside [0, min(max_seq_len, 128 * max_blocks_per_seq)].
__global__ void __launch_bounds__(1024) paged_schedule(const PagedParams p) {
    __shared__ int count[17], offset[17];
    grid_launch_dependents();  // the decode grid sets up while this runs
    const int bps = p.blocks_per_split;
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * kBlk);
    if (threadIdx.x <= 16) count[threadIdx.x] = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
        int L = p.seq_lens[s];
        if (L < 0 || L > cap) {
            if (p.status) atomicOr(p.status, kDevBadSeqlen);
            L = L < 0 ? 0 : cap;
        }
        const int nblk = (L + kBlk - 1) / kBlk;
        if (nblk / bps) atomicAdd(&count[bps], nblk / bps);
        if (nblk % bps) atomicAdd(&count[nblk % bps], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int at = 0;
        for (int b = 16; b >= 1; --b) {
            offset[b] = at;
            at += count[b];
        }
        p.sched[0] = 0;
        p.sched[1] = at;
    }
    __syncthreads();
    for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
        int L = p.seq_lens[s];
        L = L < 0 ? 0 : (L > cap ? cap : L);
        const int nblk = (L + kBlk - 1) / kBlk;
        const int nfull = nblk / bps;
        if (nfull) {
            const int at = atomicAdd(&offset[bps], nfull);
            for (int i = 0; i < nfull; ++i)
                p.pairs[at + i] = make_int4(s, i, i * bps * kBlk, min(L, (i + 1) * bps * kBlk));
        }
        if (nblk % bps) {
            const int at = atomicAdd(&offset[nblk % bps], 1);
            p.pairs[at] = make_int4(s, nfull, nfull * bps * kBlk, L);
        }
    }
}

// Merge the split partials of each (sequence, query head).
__global__ void __launch_bounds__(128) paged_combine(const PagedParams p, int D) {
    grid_dependency_wait();  // launched behind the decode grid, whose partials it reads
    const int s = blockIdx.x / p.Hq, h = blockIdx.x % p.Hq;
    int L = p.seq_lens[s];
    const int cap = min(p.max_seq_len, p.max_blocks_per_seq * kBlk);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int nsp = (L + p.blocks_per_split * kBlk - 1) / (p.blocks_per_split * kBlk);
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
    PagedPlan pl{1, 0, 0, 0, 0, 0};
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
    pl.o_bytes = (rows * D * 4 + 255) & ~size_t(255);
    pl.lse_bytes = (rows * 4 + 255) & ~size_t(255);
    pl.pairs_bytes = (static_cast<size_t>(num_seqs) * pl.max_splits * 16 + 255) & ~size_t(255);
    pl.workspace_bytes = pl.o_bytes + pl.lse_bytes + pl.pairs_bytes + 256;
    return pl;
}

int paged_slice_rows(int D) { return D <= 128 ? 128 : 64; }

template <class C>
static cudaError_t launch_paged_cfg(const CUtensorMap& tm, const PagedParams& p, int num_sms, cudaStream_t st) {
    static bool attr_done[64];  // the attribute is per function and device
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(paged_decode_sm103a<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const int n_hgroups = p.Hkv * (p.group / p.heads_per_cta);
    const long long n_items = static_cast<long long>(p.num_seqs) * n_hgroups * p.max_splits;
    const int grid = static_cast<int>(n_items < num_sms ? n_items : num_sms);
    paged_schedule<<<1, 1024, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // The decode and combine grids are programmatic dependents of the grid
    // before them: they may start while it runs and wait for it
    // (griddepcontrol.wait) before they read what it writes.
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(32 * kWarps);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, paged_decode_sm103a<C>, tm, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(p.num_seqs * p.Hq));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, paged_combine, p, static_cast<int>(C::D));
    if (e != cudaSuccess) return e;
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
