// prefill.cu -- fused attention forward for sm_103a (dense and packed varlen).
//
// For each query tile (128 rows of one document and query head):
//   S_j = Q K_j^T          tcgen05.mma, bf16 x bf16 -> fp32 in TMEM
//   P_j = exp2(S_j*c - m)  softmax warps, one thread per query row (TMEM lane)
//   O  += P_j V_j          tcgen05.mma, O accumulated in TMEM
//   out = O / l, lse = (m + log2 l) ln 2
// This is the online-softmax form of the plain definition (vllm-omni
// flash_attn.py, FlashAttentionImpl: flash_attn_func / flash_attn_varlen_func
// with softmax_scale and causal; the (out, lse) pair of _unwrap_flash_output).
//
// Two kernels:
//   fmha2_fwd_sm103a (D = 64, 96, 128): two query tiles per CTA that share
//     every K/V tile, two softmax warpgroups taking turns with the tensor
//     cores, P written back into TMEM and read by the P.V product from there,
//     TMA-store epilogue, a persistent grid for dense launches of more than
//     one wave, and the partly filled last wave split along the keys over
//     thread-block clusters that merge on chip (see the comments there);
//   fmha_fwd_sm103a (D = 192, 256): one tile per CTA (two O accumulators of
//     that width do not fit in TMEM next to the S buffers), 192 threads:
//       warps 0-3  softmax + O correction + epilogue; warp w owns TMEM lanes 32w..32w+31
//       warp 4     TMA producer: Q once, then K and V in the order the MMAs
//                  read them (K_0, K_1 V_0, K_2 V_1, ...) into a ring of slots:
//                  at D = 192 three 48 KB slots, one whole K or V tile each; at
//                  D = 256 five 32 KB slots, a K tile two slots of 128 columns,
//                  a V tile two slots of 64 keys x 256 columns
//       warp 5     TMEM allocator and MMA issuer (one elected lane)
//     S double-buffered in TMEM (S_{j+1} is issued before PV_j, so the tensor
//     core works on the next scores while the softmax warps exponentiate the
//     current ones); P written back over S_j's buffer and read by P.V from
//     TMEM, as in the two-tile kernel.  The MMAs of each slot release it as
//     they complete, so the ring refills a slot at a time, ahead of the
//     MMAs.  K is cut along D (each slot feeds full-width N = 128 score
//     products) and P.V runs as full-width N = D products (at D = 256 V is
//     cut along the keys).  Slots are as large as the ring allows: measured
//     on this part, one SM's TMA rate grows with the bytes each barrier
//     covers (16 KB: about 21 B/cycle, 32 KB: 40, 48 KB: 57), and 16 KB
//     slots held these kernels to 1180 / 1270 TFLOP/s against 1640 / 1600
//     with these.
//
// Both kernels have a paged instantiation (PAGED): K/V tiles come from the
// paged cache through block_table (vllm-ascend attention_v1.py, chunked
// prefill and speculative decode over the cache), and the two-tile kernel
// can pack a GQA group into a tile (128 / group tokens x group heads per 128
// rows).  In every mode the V rows of a document's last KV tile that lie past
// its last key are zeroed in shared memory before P.V, so a document's result
// never depends on the bytes of its neighbours (no cross-document attention,
// FlashAttentionImpl._forward_varlen_packed), NaN or not.
//
// Causal masking is bottom-right aligned (FlashAttentionImpl.forward_fa_npu:
// key kp is blocked for query qp iff kp > qp + Sk - Sq); KV tiles past the
// last visible key of the tile's last row are never loaded.
//
// Shared-memory operand layout: every operand is a stack of 64-column
// chunks, each chunk [rows x 128 B] with the 128-byte swizzle that TMA
// writes (16-byte piece c of row r at position c ^ (r % 8)).  Q and K are
// K-major operands; V is the MN-major B operand of P V.  P never touches
// shared memory in either kernel (it goes from the softmax threads to TMEM).
// Output staged for TMA stores uses the same swizzle, 128-byte boxes of
// columns.
#include <math.h>
#include <algorithm>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {

template <int D_, int BN_, int SLOTS_, int SCH_>
struct PrefillCfg {
    static constexpr int D = D_;
    static constexpr int BN = BN_;
    static constexpr int SLOTS = SLOTS_;                // K/V ring slots
    static constexpr int SCH = SCH_;                    // 64-column chunks of a K tile per slot
    static constexpr int BM = 128;
    static constexpr int NCH = (D + 63) / 64;           // 64-column chunks per row
    static constexpr int Q_BYTES = NCH * BM * 128;
    static constexpr int SLOT_BYTES = SCH * BN * 128;
    static constexpr int K_SLOTS = NCH / SCH;           // slots of one K tile
    // V cut along the keys (VR keys x D per slot) when that fills a slot, else
    // into 64-column chunks like K
    static constexpr bool VKEYS = 32 * SCH * D * 2 == SLOT_BYTES;
    static constexpr int VR = VKEYS ? 32 * SCH : BN;    // keys of a V tile per slot
    static constexpr int V_SLOTS = VKEYS ? BN / VR : K_SLOTS;
    static constexpr int V_SLOT_BYTES = VKEYS ? VR * D * 2 : SLOT_BYTES;
    static constexpr int NUM_BARS = 2 * SLOTS + 6;
    static constexpr int SMEM_BYTES = 1024 + Q_BYTES + SLOTS * SLOT_BYTES + NUM_BARS * 8 + 16;
    static constexpr int TMEM_S = 0;        // S buffers at columns [0, BN) and [BN, 2BN)
    static constexpr int TMEM_O = 2 * BN;   // O at [2BN, 2BN + D)
    static constexpr int TMEM_COLS = (2 * BN + D) <= 256 ? 256 : 512;
    static_assert(2 * BN + D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(D % 32 == 0 && BN % 64 == 0, "tile shape");
    static_assert(D % 64 == 0 && BM == BN && (D / 32) * BM * 128 <= SLOTS * SLOT_BYTES, "output staging in the ring");
    static_assert(V_SLOT_BYTES == SLOT_BYTES && VR % 16 == 0 && BN % VR == 0 && NCH % SCH == 0 && K_SLOTS <= SLOTS,
                  "V slots");
    // TMA-store epilogue for full tiles: measured +6.6% at D = 192, +1.4% at D = 256
    // (against row-predicated stores from registers)
    static constexpr bool TMA_OUT = true;
};

constexpr float kLn2 = 0.6931471805599453f;

// Used length of padded batch entry b: lens[b] clamped to [0, full] (a value
// outside is flagged), or full when lens is null.
__device__ __forceinline__ int padded_len(const int32_t* lens, int b, int full, uint32_t* status, bool report) {
    if (!lens) return full;
    const int n = lens[b];
    if (n < 0 || n > full) {
        if (report && status) atomicOr(status, kDevBadSeqlen);
        return n < 0 ? 0 : full;
    }
    return n;
}
constexpr float kRescaleThreshold = 8.0f;  // log2 units: tolerate P up to 2^8 before rescaling O

template <class C, bool PAGED>
__global__ void __launch_bounds__(192, 1)
    fmha_fwd_sm103a(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const PrefillParams p) {
    constexpr int D = C::D, BN = C::BN, SLOTS = C::SLOTS, BM = C::BM, NCH = C::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sKV = sQ + C::Q_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::Q_BYTES + SLOTS * C::SLOT_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t b_q_full = smem_u32(&bars[0]);
    auto b_kv_full = [&](int s) { return smem_u32(&bars[1 + s]); };
    auto b_kv_empty = [&](int s) { return smem_u32(&bars[1 + SLOTS + s]); };
    auto b_s_full = [&](int b) { return smem_u32(&bars[1 + 2 * SLOTS + b]); };
    const uint32_t b_p_full = smem_u32(&bars[3 + 2 * SLOTS]);
    const uint32_t b_pv_done = smem_u32(&bars[4 + 2 * SLOTS]);
    const uint32_t b_drain = smem_u32(&bars[5 + 2 * SLOTS]);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ------------------------------------------------------------ tile coordinates
    const int tile = p.causal ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;  // heavy causal tiles first
    const int h = blockIdx.y;
    const int doc = blockIdx.z;
    const int kvh = h / p.group;
    int q_start, Lq, k_start, Lk;
    if (PAGED) {  // queries packed by cu_q, keys in the paged cache
        q_start = p.cu_q[doc];
        const int q_end = p.cu_q[doc + 1];
        Lq = q_end - q_start;
        k_start = 0;
        Lk = p.seq_lens[doc];
        const bool bad = q_start < 0 || Lq < 0 || q_end > p.Tq || Lq > p.max_seqlen_q || Lk < 0 ||
                         Lk > p.max_seqlen_k || Lk > p.max_blocks * BN;
        if (bad) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0 && p.status) atomicOr(p.status, kDevBadSeqlen);
            return;
        }
    } else if (p.cu_q) {
        q_start = p.cu_q[doc];
        k_start = p.cu_k[doc];
        const int q_end = p.cu_q[doc + 1], k_end = p.cu_k[doc + 1];
        Lq = q_end - q_start;
        Lk = k_end - k_start;
        const bool bad = q_start < 0 || Lq < 0 || q_end > p.Tq || k_start < 0 || Lk < 0 ||
                         k_end > p.Tk || Lq > p.max_seqlen_q || Lk > p.max_seqlen_k;
        if (bad) {
            if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0 && p.status) atomicOr(p.status, kDevBadSeqlen);
            return;
        }
    } else {
        q_start = doc * p.Sq;
        Lq = p.Sq;
        k_start = doc * p.Sk;
        Lk = p.Sk;
    }
    // Padded batch (lens_q / lens_k): entry doc uses its first Lqu query rows
    // and Lk keys; the rows past Lqu see no key (out 0, lse -inf).
    int Lqu = Lq;
    if (!PAGED && !p.cu_q && (p.lens_q || p.lens_k)) {
        Lqu = padded_len(p.lens_q, doc, Lq, p.status, threadIdx.x == 0);
        Lk = padded_len(p.lens_k, doc, Lk, p.status, threadIdx.x == 0);
    }
    const int q0 = tile * BM;
    if (q0 >= Lq) return;  // CTA-uniform, before any barrier or TMEM use
    if (status_has_timeout(p.status, kDevTimeout)) return;
    const int diag = Lk - Lqu;
    int kend = q0 < Lqu ? Lk : 0;
    if (p.causal && q0 < Lqu) kend = min(Lk, min(q0 + BM - 1, Lqu - 1) + diag + 1);
    const int n_kv = kend > 0 ? (kend + BN - 1) / BN : 0;

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(b_kv_full(s), 1);
            mbar_init(b_kv_empty(s), 1);
        }
        mbar_init(b_s_full(0), 1);
        mbar_init(b_s_full(1), 1);
        mbar_init(b_p_full, 128);
        mbar_init(b_pv_done, 1);
        mbar_init(b_drain, 1);
        *abort_flag = p.give_up ? 1 : 0;  // 1: give up every wait (failure-path test)
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
            for (int c = 0; c < NCH; ++c) tma_load_3d(sQ + c * BM * 128, &tmQ, b_q_full, c * 64, h, q_start + q0);
            // Load t of the MMAs' order: K_0, then K_{j+1} and V_j for each j,
            // V_{n-1} last.  Chunk g of the sequence goes to slot g % SLOTS.
            int issued = 0;
            for (int t = 0; ok && t < 2 * n_kv; ++t) {
                const bool isv = t == 2 * n_kv - 1 || (t > 0 && (t & 1) == 0);
                const int jt = isv ? (t == 2 * n_kv - 1 ? n_kv - 1 : t / 2 - 1) : (t + 1) / 2;
                const CUtensorMap* m = isv ? &tmV : &tmK;
                int row = k_start + jt * BN;
                if (PAGED) {  // cache block of KV tile jt; a bad entry is flagged, block 0 read
                    int blk = p.block_table[static_cast<long long>(doc) * p.max_blocks + jt];
                    if (blk < 0 || blk >= p.num_blocks) {
                        if (p.status) atomicOr(p.status, kDevBadIndex);
                        blk = 0;
                    }
                    row = (isv ? p.num_blocks + blk : blk) * BN;
                }
                for (int q = 0; q < (isv ? C::V_SLOTS : C::K_SLOTS); ++q) {
                    const int s = issued % SLOTS, u = issued / SLOTS;
                    if (u > 0 && !mbar_wait(b_kv_empty(s), (u - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sKV + s * C::SLOT_BYTES;
                    if (isv && C::VKEYS) {  // keys [q VR, q VR + VR): NCH blocks of 64 columns (V map box: VR rows)
                        mbar_arrive_expect_tx(b_kv_full(s), C::V_SLOT_BYTES);
                        for (int c = 0; c < NCH; ++c)
                            tma_load_3d(dst + c * (C::VR * 128), m, b_kv_full(s), c * 64, kvh, row + q * C::VR);
                    } else {    // columns [64 SCH q, 64 SCH (q + 1)) of all BN keys
                        mbar_arrive_expect_tx(b_kv_full(s), C::SLOT_BYTES);
                        for (int i = 0; i < C::SCH; ++i)
                            tma_load_3d(dst + i * (BN * 128), m, b_kv_full(s), (q * C::SCH + i) * 64, kvh, row);
                    }
                    ++issued;
                }
            }
            if (!ok || *abort_flag) {
                // Let every copy this thread started land before the CTA retires.
                mbar_wait_drain(b_q_full, 0);
                for (int g = (issued > SLOTS ? issued - SLOTS : 0); g < issued; ++g)
                    mbar_wait_drain(b_kv_full(g % SLOTS), (g / SLOTS) & 1);
            }
        }
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        // Whole warp walks the schedule (warp-uniform waits and descriptor
        // arithmetic); one elected lane issues each tcgen05 instruction.
        constexpr uint32_t kIdS = idesc_bf16_f32(BM, BN, false, false);
        constexpr uint32_t kIdO = idesc_bf16_f32(BM, D, false, true);
        const bool leader = elect_one();
        const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
        const uint64_t dK = sdesc_sw128(sKV, 16, 1024);
        // V operand: VR-key blocks of 64 columns (VKEYS), or the tile's column
        // chunks in consecutive slots
        const uint64_t dV = sdesc_sw128(sKV, C::VKEYS ? C::VR * 128 : BN * 128, 1024);
        constexpr uint32_t kIdO64 = idesc_bf16_f32(BM, 64, false, true);
        auto wait_all = [&](uint32_t bar, uint32_t ph) {
            return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort_flag));
        };
        // Slots are read in the producer's order; cs / cph: the next one's slot and phase.
        int cs = 0;
        uint32_t cph = 0;
        auto next_slot = [&]() {
            if (++cs == SLOTS) {
                cs = 0;
                cph ^= 1u;
            }
        };
        auto issue_s = [&](int j) -> bool {
            const uint32_t dS = tmem + C::TMEM_S + (j & 1) * BN;
#pragma unroll 1
            for (int q = 0; q < C::K_SLOTS; ++q) {
                if (!wait_all(b_kv_full(cs), cph)) return false;
                tc_fence_after();
                if (leader) {
                    const uint64_t b0 = dK + static_cast<uint64_t>(cs * (C::SLOT_BYTES >> 4));
#pragma unroll
                    for (int i = 0; i < C::SCH; ++i)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(dS, dQ + ((((q * C::SCH + i) * BM) * 128 + kk * 32) >> 4),
                                        b0 + ((i * BN * 128 + kk * 32) >> 4), kIdS, (q > 0 || i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(b_kv_empty(cs));
                }
                __syncwarp();
                next_slot();
            }
            if (leader) mma_commit(b_s_full(j & 1));
            __syncwarp();
            return true;
        };
        // A launch told to give up (p.give_up) stops here, before any MMA; the
        // other warps' waits then never complete and run out at once.
        ok = !*abort_flag && wait_all(b_q_full, 0);
        if (ok && n_kv > 0) ok = issue_s(0);
        for (int j = 0; ok && j < n_kv; ++j) {
            if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
            if (!(ok = wait_all(b_p_full, j & 1))) break;
            // O += P_j V_j; P_j (bf16 pairs) read from the first BN / 2 columns
            // of S_j's buffer.  Rows past the document's last key (the next
            // document's, the next batch entry's, or cache slots past
            // seq_len) may hold anything, NaN included; P is 0 there but
            // 0 * NaN is not, so V rows past the end are zeroed first.
            const uint32_t a = tmem + C::TMEM_S + (j & 1) * BN;
            const int lim = Lk - j * BN;  // keys of this tile inside the document
            if (C::VKEYS) {
#pragma unroll 1
                for (int q = 0; q < C::V_SLOTS; ++q) {
                    if (!(ok = wait_all(b_kv_full(cs), cph))) break;
                    const uint32_t vb = sKV + cs * C::SLOT_BYTES;
                    const int ql = lim - q * C::VR;  // keys of this slot inside the document
                    if (ql < C::VR) {
                        const int r0 = ql > 0 ? ql : 0;
                        for (int idx = lane; idx < (C::VR - r0) * NCH * 8; idx += 32) {
                            const int u = idx & 7, rc = idx >> 3, c = rc % NCH, rr = r0 + rc / NCH;
                            st_shared_v4(vb + c * (C::VR * 128) + rr * 128 + u * 16, 0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    tc_fence_after();
                    if (leader) {
                        const uint64_t b0 = dV + static_cast<uint64_t>(cs * (C::SLOT_BYTES >> 4));
#pragma unroll
                        for (int kk = 0; kk < C::VR / 16; ++kk)
                            mma_bf16_ts(tmem + C::TMEM_O, a + (q * (C::VR / 16) + kk) * 8,
                                        b0 + ((kk * 16 * 128) >> 4), kIdO, (j > 0 || q > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(b_kv_empty(cs));
                    }
                    __syncwarp();
                    next_slot();
                }
            } else if (cs + C::V_SLOTS <= SLOTS) {
                // the tile's chunks lie in slots cs .. cs + V_SLOTS - 1 (one
                // phase), chunk c at sKV + cs SLOT_BYTES + c BN 128
#pragma unroll 1
                for (int q = 0; ok && q < C::V_SLOTS; ++q) ok = wait_all(b_kv_full(cs + q), cph);
                if (!ok) break;
                if (lim < BN) {
                    for (int idx = lane; idx < (BN - lim) * NCH * 8; idx += 32) {
                        const int u = idx & 7, rc = idx >> 3, c = rc % NCH, rr = lim + rc / NCH;
                        st_shared_v4(sKV + cs * C::SLOT_BYTES + c * (BN * 128) + rr * 128 + u * 16, 0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (leader) {
                    const uint64_t b0 = dV + static_cast<uint64_t>(cs * (C::SLOT_BYTES >> 4));
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_bf16_ts(tmem + C::TMEM_O, a + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdO,
                                    (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int q = 0; q < C::V_SLOTS; ++q) mma_commit(b_kv_empty(cs + q));
                }
                __syncwarp();
                for (int q = 0; q < C::V_SLOTS; ++q) next_slot();
            } else {
                // the tile wraps around the ring: one N = 64 product per chunk
#pragma unroll 1
                for (int q = 0; q < C::V_SLOTS; ++q) {
                    if (!(ok = wait_all(b_kv_full(cs), cph))) break;
                    const uint32_t vb = sKV + cs * C::SLOT_BYTES;
                    if (lim < BN) {
                        for (int idx = lane; idx < (BN - lim) * C::SCH * 8; idx += 32) {
                            const int u = idx & 7, rc = idx >> 3, i = rc % C::SCH, rr = lim + rc / C::SCH;
                            st_shared_v4(vb + i * (BN * 128) + rr * 128 + u * 16, 0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    tc_fence_after();
                    if (leader) {
#pragma unroll
                        for (int i = 0; i < C::SCH; ++i) {
                            const uint64_t b0 = dV + static_cast<uint64_t>((cs * C::SLOT_BYTES + i * BN * 128) >> 4);
#pragma unroll
                            for (int kk = 0; kk < BN / 16; ++kk)
                                mma_bf16_ts(tmem + C::TMEM_O + (q * C::SCH + i) * 64, a + kk * 8,
                                            b0 + ((kk * 16 * 128) >> 4), kIdO64, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(b_kv_empty(cs));
                    }
                    __syncwarp();
                    next_slot();
                }
            }
            if (!ok) break;
            if (leader) mma_commit(b_pv_done);
            __syncwarp();
        }
        // Everything issued above must finish before TMEM is released.
        if (leader) mma_commit(b_drain);
        __syncwarp();
        mbar_wait_drain(b_drain, 0);
    } else {
        // ------------------------------------------------------------- softmax
        const int r = threadIdx.x;  // row within the tile == TMEM lane
        const int row = q0 + r;     // row within the document
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        // keys [0, row_lim) visible
        const int row_lim = row >= Lqu ? 0 : (p.causal ? min(Lk, row + diag + 1) : Lk);
        const float c2 = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < n_kv; ++j) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_s_full(j & 1), (j >> 1) & 1, abort_flag)))) break;
            tc_fence_after();
            uint32_t sr[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
                tmem_ld32(tl + C::TMEM_S + (j & 1) * BN + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
            tmem_wait_ld();
            const int kbase = j * BN;
            const bool edge = (kbase + BN > Lk) || (p.causal && kbase + BN - 1 > q0 + diag) || q0 + BM > Lqu;
            if (edge) {
                const int lim = row_lim - kbase;
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
            }
            // row max: three-input max into 4 independent chains (16 deep, 2 values per op)
            float mxp[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) mxp[i] = __uint_as_float(sr[i]);
#pragma unroll
            for (int c = 4; c < BN; c += 2)
                mxp[(c >> 1) & 3] = fmax3(mxp[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            const float mx = fmaxf(fmax3(mxp[0], mxp[1], mxp[2]), mxp[3]);
            const float m_new = fmaxf(m, mx * c2);
            const bool need = m_new > m + kRescaleThreshold;
            const bool warp_need = __any_sync(0xffffffffu, need);
            float alpha = 1.f;
            if (warp_need && m_new > m) {
                alpha = ex2(m - m_new);
                m = m_new;
            }
            l *= alpha;
            // O must hold PV_{j-1} before it is rescaled.  S_j was issued after
            // PV_{j-2} only, so here PV_0 .. PV_{j-2} are complete and PV_j not
            // yet issued: pv_done has completed j - 1 or j phases, and a wait
            // on the parity of phase j - 1 is exact whichever it is.  It is
            // made when O is rescaled, and on the last step, so that after the
            // loop pv_done is again within one phase of the final wait.  P_j
            // goes over S_j's own buffer, whose previous P (P_{j-2}) PV_{j-2}
            // read before S_j was written.
            if (j > 0 && (warp_need || j + 1 == n_kv)) {
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
            // P = 2^(S c - m) as bf16 pairs over the first BN / 2 columns of S_j
            const float msub = (m == -INFINITY) ? 0.f : m;
            const float2 c2x2 = make_float2(c2, c2), negm = make_float2(-msub, -msub);
            float2 rsp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};  // independent partial row sums, in pairs
            const uint32_t tS = tl + C::TMEM_S + (j & 1) * BN;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 t = __ffma2_rn(
                        make_float2(__uint_as_float(sr[c * 32 + e]), __uint_as_float(sr[c * 32 + e + 1])), c2x2, negm);
                    const float2 pp = make_float2(ex2(t.x), ex2(t.y));
                    rsp[(e >> 1) & 3] = __fadd2_rn(rsp[(e >> 1) & 3], pp);
                    pk[e >> 1] = pack_bf16x2(pp.x, pp.y);
                }
                tmem_st16(tS + c * 16, pk);
            }
            const float2 rr = __fadd2_rn(__fadd2_rn(rsp[0], rsp[1]), __fadd2_rn(rsp[2], rsp[3]));
            l += rr.x + rr.y;
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
        if (C::TMA_OUT && q0 + BM <= Lq) {
            // A tile wholly inside its document leaves through shared memory:
            // rows staged in the TMA 128-byte-swizzled box layout in 16 KB
            // slots of the K/V area (free: PV of the last KV tile was the last
            // MMA) and written by tiled TMA stores.
            const bool f32 = p.out_f32 != 0;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const int boxes = f32 ? D / 32 : D / 64, cols = f32 ? 32 : 64;  // 128-byte boxes per row
            const int sw = r & 7;
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
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
                if (f32) {  // 32 columns = one 128-byte box row
                    const uint32_t rb = sKV + c * (BM * 128) + r * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(rb + ((k ^ sw) << 4), o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                } else {    // 32 columns = half a box row
                    const uint32_t rb = sKV + (c >> 1) * (BM * 128) + r * 128;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_shared_v4(rb + ((((c & 1) * 4 + k) ^ sw) << 4),
                                     pack_bf16x2(__uint_as_float(o[8 * k]), __uint_as_float(o[8 * k + 1])),
                                     pack_bf16x2(__uint_as_float(o[8 * k + 2]), __uint_as_float(o[8 * k + 3])),
                                     pack_bf16x2(__uint_as_float(o[8 * k + 4]), __uint_as_float(o[8 * k + 5])),
                                     pack_bf16x2(__uint_as_float(o[8 * k + 6]), __uint_as_float(o[8 * k + 7])));
                }
            }
            fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine
            named_bar_sync(1, 128);
            if (r == 0) {
                for (int b = 0; b < boxes; ++b) tma_store_3d(&tmO, sKV + b * (BM * 128), b * cols, h, q_start + q0);
                bulk_commit();
                bulk_wait_read0();  // the staging area must outlive the reads
            }
            if (ok && p.lse) {
                const long long lrow = p.lse_row_global ? (q_start + row) : row;
                p.lse[doc * p.lse_bstride + h * p.lse_hstride + lrow] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
            }
        } else {
        const bool row_valid = ok && row < Lq;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const long long orow = static_cast<long long>(q_start + row) * p.Hq + h;
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
                    float* dst = reinterpret_cast<float*>(p.out) + orow * D + c * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        st_global_v4(dst + e, __float_as_uint(__uint_as_float(o[e]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 1]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 2]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 3]) * inv_l));
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + orow * D + c * 32;
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
        if (row_valid && p.lse) {
            const long long lrow = p.lse_row_global ? (q_start + row) : row;
            p.lse[doc * p.lse_bstride + h * p.lse_hstride + lrow] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        }
        }
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

// ---------------------------------------------------------------------------
// Two query tiles per CTA (D <= 128).
//
// An item is 256 query rows of one (document, head): tile A = rows
// [q0, q0 + 128), tile B = [q0 + 128, q0 + 256).  Each tile has its own
// softmax warpgroup (warps 0-3: A, warps 4-7: B), so while one warpgroup
// exponentiates its scores the tensor core runs the other tile's products.
//   warp 8   TMA producer (per item Q_A, Q_B; then K_0 V_0 K_1 V_1 ...)
//   warp 9   TMEM allocator + MMA issuer, in the order
//            S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//   warps 10-11 idle (they complete the third warpgroup)
// A CTA runs one item, or (persistent launches) several in turn: the ring
// of K/V stages, the mbarrier phases and the Q buffers carry on from item
// to item; Q of the next item is loaded once the current item's last S
// products are done, its K_0 while the current epilogue runs.
// Registers: launched at 168 per thread; the third warpgroup gives back
// down to 88 so each softmax thread can hold a whole 128-column S row (208).
// TMEM: S_A [0,128) S_B [128,256) O_A [256, 256+D) O_B [256+D, 256+2D).
// P_X (bf16 pairs) is written back over the first 64 columns of S_X and
// read from there by the P.V product (tcgen05.mma with A in tensor memory),
// so P never goes through shared memory.  The MMA thread issues every
// tcgen05.mma in order, so once S_X(j) is complete PV_X(j-1) is complete
// too: the softmax warps may then rescale O_X and overwrite P_X without a
// separate wait.
// Most documents a persistent varlen launch walks (beyond: one CTA per item).
constexpr int kWalkMaxDocs = 512;

template <int D_, int STAGES_>
struct Prefill2Cfg {
    static constexpr int D = D_;
    static constexpr int BN = 128;
    static constexpr int STAGES = STAGES_;
    static constexpr int BM = 128;  // rows per tile; two tiles per CTA
    static constexpr int NCH = (D + 63) / 64;
    static constexpr int QT_BYTES = NCH * BM * 128;  // one Q tile
    static constexpr int KV_BYTES = NCH * BN * 128;
    static constexpr int NUM_BARS = 2 * STAGES + 11;
    // + 16 bytes: TMEM address and abort flag; + 12 x 16: each warp's cursor of the persistent varlen walk
    static constexpr int SMEM_BYTES = 1024 + 2 * QT_BYTES + STAGES * KV_BYTES + NUM_BARS * 8 + 16 + 12 * 16;
    static constexpr int TMEM_S = 0;          // S_X at X * BN
    static constexpr int TMEM_O = 2 * BN;     // O_X at TMEM_O + X * D
    static constexpr int TMEM_COLS = 512;
    // setmaxnreg split of the 384 x 168 launched registers: softmax warpgroups
    // / producer + MMA warpgroup (with the item walk of packed documents the
    // MMA and producer code needs more than 72; the softmax code fits in 208)
    static constexpr int REG_SOFTMAX = 208;
    static constexpr int REG_OTHER = 88;
    static_assert(2 * 128 * REG_SOFTMAX + 128 * REG_OTHER <= 384 * 168, "register split");
    static_assert(2 * BN + 2 * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(2 * BM * D * 4 <= STAGES * KV_BYTES && 2 * BM * 8 <= 2 * QT_BYTES, "split-merge staging");
    static_assert(KV_BYTES == NCH * BM * 128 && STAGES >= 3, "output staging stages");
};

// Merge of an item split along the keys over a cluster of p.split CTAs (the
// softmax threads of every CTA call this; the other warps only pass the same
// three cluster barriers).  CTA c holds, for the pair's 256 rows, O_c
// (unnormalised, in TMEM), m_c and l_c over its key range; the partial
// softmaxes combine as
//   out = sum_c 2^(m_c - M) O_c / L,   L = sum_c 2^(m_c - M) l_c,   M = max_c m_c,
//   lse = (M + log2 L) ln 2.
// Each CTA stages its weighted rows in its own shared memory; CTA c then sums
// rows [c R, (c + 1) R), R = 256 / p.split, over the cluster through
// distributed shared memory and writes them.  Called once every MMA of the
// CTA has completed, so the Q and K/V areas are free.
template <int D>
__device__ __forceinline__ void split_merge(uint8_t* smem, uint32_t sO, uint32_t tO, int pr, float m, float l,
                                            bool have_o, bool ok, int crank, int q0, int Lq, int q_start, int h,
                                            int doc, const PrefillParams& p) {
    constexpr int ROWS = 256, CH = D / 4;  // 16-byte chunks per staged fp32 row
    const int C = p.split;
    float2* sML = reinterpret_cast<float2*>(smem);  // (m, l) of the 256 rows, over the Q area
    sML[pr] = make_float2(m, l);
    cluster_sync();
    auto merged = [&](int row, float& M, float& L) {
        float mc[8], lc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            mc[c] = -INFINITY;
            lc[c] = 0.f;
            if (c < C) {
                const float2 v = ld_cluster_f2(mapa_shared(smem_u32(&sML[row]), c));
                mc[c] = v.x;
                lc[c] = v.y;
            }
        }
        M = mc[0];
#pragma unroll
        for (int c = 1; c < 8; ++c) M = fmaxf(M, mc[c]);
        L = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            if (lc[c] > 0.f) L += lc[c] * ex2(mc[c] - M);
    };
    float M, L;
    merged(pr, M, L);
    const float w = (L > 0.f && l > 0.f) ? ex2(m - M) / L : 0.f;
    const uint32_t row_base = sO + static_cast<uint32_t>(pr) * (D * 4);
#pragma unroll 1
    for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t o[32];
        if (have_o && ok) {
            tmem_ld32(tO + c32 * 32, o);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
            const int slot = (c32 * 8 + e4) ^ (pr & 7);
            st_shared_v4(row_base + slot * 16, __float_as_uint(__uint_as_float(o[4 * e4]) * w),
                         __float_as_uint(__uint_as_float(o[4 * e4 + 1]) * w),
                         __float_as_uint(__uint_as_float(o[4 * e4 + 2]) * w),
                         __float_as_uint(__uint_as_float(o[4 * e4 + 3]) * w));
        }
    }
    cluster_sync();
    const int R = ROWS / C;
    const int t = static_cast<int>(threadIdx.x);  // 0 .. 255
#pragma unroll 1
    for (int id = t; id < R * CH; id += ROWS) {
        const int orow = crank * R + id / CH, ch = id % CH;
        const uint32_t off = sO + static_cast<uint32_t>(orow) * (D * 4) + static_cast<uint32_t>((ch ^ (orow & 7)) * 16);
        float4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = c < C ? ld_cluster_f4(mapa_shared(off, c)) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 acc = v[0];
#pragma unroll
        for (int c = 1; c < 8; ++c) {
            acc.x += v[c].x;
            acc.y += v[c].y;
            acc.z += v[c].z;
            acc.w += v[c].w;
        }
        const int qrow = q0 + orow;
        if (ok && qrow < Lq) {
            const long long o_off = (static_cast<long long>(q_start + qrow) * p.Hq + h) * D + ch * 4;
            if (p.out_f32)
                st_global_v4(reinterpret_cast<float*>(p.out) + o_off, __float_as_uint(acc.x), __float_as_uint(acc.y),
                             __float_as_uint(acc.z), __float_as_uint(acc.w));
            else
                *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + o_off) =
                    make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        }
    }
    if (t < R && p.lse) {
        const int orow = crank * R + t, qrow = q0 + orow;
        float Mr, Lr;
        merged(orow, Mr, Lr);
        if (ok && qrow < Lq) {
            const long long lrow = p.lse_row_global ? (q_start + qrow) : qrow;
            p.lse[doc * p.lse_bstride + h * p.lse_hstride + lrow] = Lr > 0.f ? (Mr + __log2f(Lr)) * kLn2 : -INFINITY;
        }
    }
    cluster_sync();  // no CTA leaves while another still reads its shared memory
}

// DEFER (dense launches of few KV tiles): the wait for the last staged
// stores' reads, and the b_staged arrival, move from the end of the epilogue
// to after the next item's first P hand-over, where they rarely wait.  Its
// own instantiation: the extra code in the step loop costs the long-item
// launches a little.
template <class C, bool PAGED, bool WALK, bool DEFER = false>
__global__ void __launch_bounds__(384, 1)
    fmha2_fwd_sm103a(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const PrefillParams p) {
    constexpr int D = C::D, BN = C::BN, STAGES = C::STAGES, BM = C::BM, NCH = C::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sQ = smem_u32(smem);  // Q_X at sQ + X * QT_BYTES
    const uint32_t sKV = sQ + 2 * C::QT_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * C::QT_BYTES + STAGES * C::KV_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t b_q_full = smem_u32(&bars[0]);
    auto b_kv_full = [&](int s) { return smem_u32(&bars[1 + s]); };
    auto b_kv_empty = [&](int s) { return smem_u32(&bars[1 + STAGES + s]); };
    auto b_s_full = [&](int x) { return smem_u32(&bars[1 + 2 * STAGES + x]); };
    auto b_p_full = [&](int x) { return smem_u32(&bars[3 + 2 * STAGES + x]); };
    auto b_pv_done = [&](int x) { return smem_u32(&bars[5 + 2 * STAGES + x]); };
    const uint32_t b_drain = smem_u32(&bars[7 + 2 * STAGES]);
    const uint32_t b_q_empty = smem_u32(&bars[8 + 2 * STAGES]);  // Q tiles read by every S of an item
    // persistent: tile X's output staging has been read by its TMA stores
    auto b_staged = [&](int x) { return smem_u32(&bars[9 + 2 * STAGES + x]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ------------------------------------------------------------ work items
    // An item is one pair of query tiles of one (head, document).  Varlen:
    // the CTA's grid cell (tile, head, document).  Dense: item item_base +
    // blockIdx.x (of blockIdx.x / split in a split cluster), or, persistent,
    // items item_base + blockIdx.x + i * gridDim.x below item_end, one after
    // the other: the next item's Q and K/V loads and first S products then
    // overlap the current item's softmax tail and epilogue.
    const bool split = p.split > 1;  // kernel-uniform
    // GQA packing (paged prefill): a tile's 128 rows are TPT tokens x the
    // group's query heads, row r = token r / group, head r % group.
    const int gq = (PAGED && p.gqa_pack) ? p.group : 1;
    const int TPT = BM / gq;
    const bool persist = p.persist != 0;
    const int crank = split ? static_cast<int>(cluster_ctarank()) : 0;
    struct Item {
        int h, doc, kvh, q_start, Lq, Lqu, k_start, Lk, q0, diag, nA, nB, nmax, j0;  // Lqu: used query rows
        bool valid;  // false: no such item, or one with nothing to do (CTA-uniform)
    };
    // Persistent varlen walk (linear == 2).  The items are listed tile-major:
    // level r holds tile t = T - 1 - r (T = tile pairs of the longest
    // document) of every document that has it, heads fastest, so the heavy
    // causal tiles come first across all documents.  CTA b takes list
    // positions k * G + b (k even) and k * G + G - 1 - b (k odd), G CTAs: a
    // snake over the list that keeps the CTAs' loads within a few percent of
    // each other.  Each role walks the list with its own cursor (positions
    // only grow); a document with inconsistent cu_seqlens has no tiles, and
    // CTA 0 reports it.
    // A cursor is three ints in shared memory, one per warp, so that it holds
    // no register in the softmax loop: {level, documents in the level (-1:
    // not started), list position of the level's first item (the host keeps
    // the list under 2^31)}.  The lanes in `mask` (every lane of the warp, or
    // lane 0 alone for the producer) read and write it together, between
    // __syncwarp(mask), so they always see the same values.
    struct Walk {
        volatile int* c;
        unsigned mask;
    };
    auto walk_here = [&](unsigned mask) {
        Walk W{reinterpret_cast<volatile int*>(tmem_slot + 4) + 4 * (threadIdx.x >> 5), mask};
        if (WALK) {
            W.c[1] = -1;
            __syncwarp(mask);
        }
        return W;
    };
    const int walk_T = (p.max_seqlen_q + 2 * BM - 1) / (2 * BM);
    auto doc_tiles = [&](int d, bool report) -> int {
        const int qs = p.cu_q[d], qe = p.cu_q[d + 1], ks = p.cu_k[d], ke = p.cu_k[d + 1];
        const bool bad = qs < 0 || qe < qs || qe > p.Tq || qe - qs > p.max_seqlen_q || ks < 0 || ke < ks ||
                         ke > p.Tk || ke - ks > p.max_seqlen_k;
        if (bad) {
            if (report && p.status) atomicOr(p.status, kDevBadSeqlen);
            return 0;
        }
        return (qe - qs + 2 * BM - 1) / (2 * BM);
    };
    auto level_docs = [&](int t, bool report) {
        int n = 0;
        for (int d = 0; d < p.num_docs; ++d) n += doc_tiles(d, report) > t ? 1 : 0;
        return n;
    };
    auto item_at = [&](int i, Walk& W) -> Item {
        Item I{};
        I.valid = false;
        int tile;
        // (the run-time test of linear keeps the register allocation of the walk
        // kernel free of spills; linear is always 2 in it)
        if (WALK && p.linear == 2) {
            const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
            const long long gl = static_cast<long long>(i) * G + ((i & 1) ? G - 1 - b : b);
            if (gl > 0x7fffffffLL) return I;
            const int g = static_cast<int>(gl);
            __syncwarp(W.mask);
            int wr = W.c[0], wn = W.c[1], wbase = W.c[2];
            __syncwarp(W.mask);
            if (wn < 0) {
                wr = 0;
                wbase = 0;
                wn = walk_T > 0 ? level_docs(walk_T - 1, blockIdx.x == 0 && threadIdx.x == 0) : 0;
            }
            bool past = false;
            while (!past && g - wbase >= wn * p.Hq) {
                wbase += wn * p.Hq;
                if (++wr >= walk_T)
                    past = true;
                else
                    wn = level_docs(walk_T - 1 - wr, false);
            }
            W.c[0] = wr;
            W.c[1] = wn;
            W.c[2] = wbase;
            __syncwarp(W.mask);
            if (past) return I;
            tile = walk_T - 1 - wr;
            const int k = g - wbase;
            int rank = k / p.Hq;
            I.h = k % p.Hq;
            I.doc = -1;
            for (int d = 0; d < p.num_docs && I.doc < 0; ++d)
                if (doc_tiles(d, false) > tile && rank-- == 0) I.doc = d;
            if (I.doc < 0) return I;
        } else if (p.linear) {
            long long item;
            if (persist)
                item = p.item_base + static_cast<long long>(blockIdx.x) + static_cast<long long>(i) * gridDim.x;
            else
                item = i == 0 ? p.item_base + static_cast<long long>(split ? blockIdx.x / p.split : blockIdx.x) : -1;
            if (item < 0 || (persist && item >= p.item_end)) return I;
            tile = static_cast<int>(item % p.tiles);
            const int hb = static_cast<int>(item / p.tiles);
            I.h = hb % p.Hq;
            I.doc = hb / p.Hq;
            if (p.causal) tile = p.tiles - 1 - tile;  // heavy causal tiles first
        } else {
            if (i > 0) return I;
            tile = p.causal ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;
            I.h = blockIdx.y * gq;  // with GQA packing blockIdx.y is the KV head
            I.doc = blockIdx.z;
        }
        I.kvh = I.h / p.group;
        if (PAGED) {  // queries packed by cu_q, keys in the paged cache
            I.q_start = p.cu_q[I.doc];
            const int q_end = p.cu_q[I.doc + 1];
            I.Lq = q_end - I.q_start;
            I.k_start = 0;
            I.Lk = p.seq_lens[I.doc];
            const bool bad = I.q_start < 0 || I.Lq < 0 || q_end > p.Tq || I.Lq > p.max_seqlen_q || I.Lk < 0 ||
                             I.Lk > p.max_seqlen_k || I.Lk > p.max_blocks * BN;
            if (bad) {
                if (threadIdx.x == 0 && blockIdx.x == 0 && I.h == 0 && p.status) atomicOr(p.status, kDevBadSeqlen);
                return I;
            }
        } else if (p.cu_q) {
            I.q_start = p.cu_q[I.doc];
            I.k_start = p.cu_k[I.doc];
            const int q_end = p.cu_q[I.doc + 1], k_end = p.cu_k[I.doc + 1];
            I.Lq = q_end - I.q_start;
            I.Lk = k_end - I.k_start;
            const bool bad = I.q_start < 0 || I.Lq < 0 || q_end > p.Tq || I.k_start < 0 || I.Lk < 0 ||
                             k_end > p.Tk || I.Lq > p.max_seqlen_q || I.Lk > p.max_seqlen_k;
            if (bad) {
                if (threadIdx.x == 0 && blockIdx.x == 0 && I.h == 0 && p.status) atomicOr(p.status, kDevBadSeqlen);
                return I;
            }
        } else {
            I.q_start = I.doc * p.Sq;
            I.Lq = p.Sq;
            I.k_start = I.doc * p.Sk;
            I.Lk = p.Sk;
        }
        // Padded batch (lens_q / lens_k): entry doc uses its first Lqu query
        // rows and Lk keys; its rows past Lqu see no key (out 0, lse -inf)
        // and its tiles wholly past Lqu load no K/V.
        I.Lqu = I.Lq;
        if (!PAGED && !WALK && !p.cu_q && (p.lens_q || p.lens_k)) {
            const bool report = threadIdx.x == 0;  // any CTA that meets a bad length flags it
            I.Lqu = padded_len(p.lens_q, I.doc, I.Lq, p.status, report);
            I.Lk = padded_len(p.lens_k, I.doc, I.Lk, p.status, report);
        }
        I.q0 = tile * 2 * TPT;
        if (I.q0 >= I.Lq) return I;
        I.diag = I.Lk - I.Lqu;
        // KV tiles each query tile needs (0 for a tile with no used rows)
        auto kv_tiles = [&](int first_row) {
            if (first_row >= I.Lqu) return 0;
            int kend = I.Lk;
            if (p.causal) kend = min(I.Lk, min(first_row + TPT - 1, I.Lqu - 1) + I.diag + 1);
            return kend > 0 ? (kend + BN - 1) / BN : 0;
        };
        I.nA = kv_tiles(I.q0);
        I.nB = kv_tiles(I.q0 + TPT);
        // A split item (non-causal, so both tiles see the same keys) gives CTA
        // `crank` of its cluster KV tiles [j0, j1); loops below count from j0.
        I.j0 = 0;
        if (split) {
            const int n = max(I.nA, I.nB);
            I.j0 = crank * n / p.split;
            const int j1 = (crank + 1) * n / p.split;
            I.nA = I.nA > 0 ? j1 - I.j0 : 0;
            I.nB = I.nB > 0 ? j1 - I.j0 : 0;
        }
        I.nmax = max(I.nA, I.nB);
        I.valid = true;
        return I;
    };
    // Whether tile x of item I leaves through staged TMA stores in the K/V
    // area in a persistent launch (the softmax warps' epilogue condition):
    // a full tile, with KV tiles, that finishes last or with the other tile.
    auto stages_output = [&](const Item& I, int x) -> bool {
        const int nx = x ? I.nB : I.nA, ny = x ? I.nA : I.nB;
        return persist && !split && I.nmax > 0 && I.q0 + (x + 1) * TPT <= I.Lq && nx >= ny;
    };
    // Before any barrier or TMEM use; never taken by a split cluster, and a
    // persistent CTA always has a first item (but for a varlen walk whose
    // list is shorter than the grid).
    {
        Walk W0 = walk_here(0xffffffffu);  // set again by each role below, after the setup barrier
        if (!item_at(0, W0).valid) return;
    }
    if (!split && status_has_timeout(p.status, kDevTimeout)) return;
    // The split last wave (launched behind this grid, independent of its
    // results) may take each SM as soon as this grid's CTA there is done.
    if (!split) grid_launch_dependents();

    // ------------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(b_kv_full(s), 1);
            mbar_init(b_kv_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_s_full(x), 1);
            mbar_init(b_p_full(x), 128);
            mbar_init(b_pv_done(x), 1);
        }
        mbar_init(b_drain, 1);
        mbar_init(b_q_empty, 1);
        mbar_init(b_staged(0), 1);
        mbar_init(b_staged(1), 1);
        *abort_flag = p.give_up ? 1 : 0;  // 1: give up every wait (failure-path test)
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    if (warp >= 8) {
      regs_dec<C::REG_OTHER>();
      if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int t = 0, nq = 0;  // K/V loads and Q loads issued, over all items
            // Tiles whose staged output the next loads must wait for, and the
            // staging phases of each tile waited so far (persistent launches).
            bool pend[2] = {false, false};
            int pend_stage[2] = {-1, -1};  // the K/V stage each pending tile's output occupies
            uint32_t staged_waits[2] = {0u, 0u};
            auto wait_staged = [&](int x) {
                ok = ok && mbar_wait(b_staged(x), staged_waits[x] & 1, abort_flag);
                ++staged_waits[x];
                pend[x] = false;
            };
            Walk W = walk_here(1u);  // lane 0 alone
            for (int i = 0; ok; ++i) {
                const Item I = item_at(i, W);
                if (!I.valid) break;
                // Q_A, Q_B of item i replace item i-1's once its S products are done
                if (i > 0 && !mbar_wait(b_q_empty, (i - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(b_q_full, 2 * C::QT_BYTES);
                for (int x = 0; x < 2; ++x)
                    for (int c = 0; c < NCH; ++c)
                        tma_load_3d(sQ + x * C::QT_BYTES + c * BM * 128, &tmQ, b_q_full, c * 64, I.h,
                                    I.q_start + I.q0 + x * TPT);
                ++nq;
                for (int tt = 0; tt < 2 * I.nmax; ++tt, ++t) {
                    const int s = t % STAGES, u = t / STAGES;
                    // An earlier item's output staged in this stage must have
                    // been read by its stores first (each tile that staged
                    // arrives once on its own barrier, so the waits meet every
                    // phase in order).
                    for (int x = 0; x < 2; ++x)
                        if (pend[x] && pend_stage[x] == s) wait_staged(x);
                    if (!ok) break;
                    if (u > 0 && !mbar_wait(b_kv_empty(s), (u - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const CUtensorMap* m = (tt & 1) ? &tmV : &tmK;
                    int row = I.k_start + (I.j0 + (tt >> 1)) * BN;
                    if (PAGED) {  // cache block of KV tile j; a bad entry is flagged, block 0 read
                        int blk = p.block_table[static_cast<long long>(I.doc) * p.max_blocks + I.j0 + (tt >> 1)];
                        if (blk < 0 || blk >= p.num_blocks) {
                            if (p.status) atomicOr(p.status, kDevBadIndex);
                            blk = 0;
                        }
                        row = ((tt & 1) ? p.num_blocks + blk : blk) * BN;
                    }
                    mbar_arrive_expect_tx(b_kv_full(s), C::KV_BYTES);
                    for (int c = 0; c < NCH; ++c)
                        tma_load_3d(sKV + s * C::KV_BYTES + c * BN * 128, m, b_kv_full(s), c * 64, I.kvh, row);
                }
                if (!ok) break;
                for (int x = 0; x < 2; ++x)
                    if (stages_output(I, x)) {
                        if (pend[x]) wait_staged(x);  // an older staging not yet passed by the loads
                        pend[x] = true;
                        pend_stage[x] = (t + STAGES - 2 + x) % STAGES;  // t: the next item's K_0
                    }
                if (!ok) break;
            }
            if (!ok || *abort_flag) {
                // Let every copy this thread started land before the CTA retires.
                if (nq > 0) mbar_wait_drain(b_q_full, (nq - 1) & 1);
                for (int tt = (t > STAGES ? t - STAGES : 0); tt < t; ++tt)
                    mbar_wait_drain(b_kv_full(tt % STAGES), (tt / STAGES) & 1);
            }
        }
    } else if (warp == 9) {
        // ----------------------------------------------------------------- MMA
        // The whole warp walks the schedule, so every wait and all descriptor
        // arithmetic stay warp-uniform; one elected lane issues each tcgen05
        // instruction.  Shared-memory descriptors are built once and offset by
        // compile-time constants; the K/V ring position advances by counters.
        constexpr uint32_t kIdS = idesc_bf16_f32(BM, BN, false, false);
        constexpr uint32_t kIdO = idesc_bf16_f32(BM, D, false, true);
        const bool leader = elect_one();
        const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
        const uint64_t dK = sdesc_sw128(sKV, 16, 1024);
        const uint64_t dV = sdesc_sw128(sKV, BN * 128, 1024);
        auto issue_s = [&](int x, int s) {  // S_X = Q_X K^T, K in stage s
            if (leader) {
                const uint64_t a0 = dQ + static_cast<uint64_t>(x * (C::QT_BYTES >> 4));
                const uint64_t b0 = dK + static_cast<uint64_t>(s * (C::KV_BYTES >> 4));
                const uint32_t d = tmem + C::TMEM_S + x * BN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t oa = ((kk >> 2) * BM * 128 + (kk & 3) * 32) >> 4;
                    const uint32_t ob = ((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4;
                    mma_bf16_ss(d, a0 + oa, b0 + ob, kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit(b_s_full(x));
            }
            __syncwarp();
        };
        auto issue_pv = [&](int x, int s, bool acc) {  // O_X += P_X V, V in stage s
            if (leader) {
                const uint64_t b0 = dV + static_cast<uint64_t>(s * (C::KV_BYTES >> 4));
                const uint32_t d = tmem + C::TMEM_O + x * D, a = tmem + C::TMEM_S + x * BN;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16_ts(d, a + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdO, (acc || kk > 0) ? 1u : 0u);
                mma_commit(b_pv_done(x));
            }
            __syncwarp();
        };
        auto release = [&](int s) {  // stage s is free once the MMAs issued so far finish
            if (leader) mma_commit(b_kv_empty(s));
            __syncwarp();
        };
        auto wait_all = [&](uint32_t bar, uint32_t ph) {
            return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort_flag));
        };
        auto adv = [](int& s, uint32_t& ph) {
            s += 2;
            if (s >= STAGES) {
                s -= STAGES;
                ph ^= 1u;
            }
        };
        int tbase = 0;             // ring index of the current item's K_0 (K_j: tbase + 2j, V_j: + 1)
        uint32_t pa = 0, pb = 0;   // softmax steps of tiles A and B in earlier items
        Walk W = walk_here(0xffffffffu);
        for (int i = 0; ok; ++i) {
            const Item I = item_at(i, W);
            if (!I.valid) break;
            const int nA = I.nA, nB = I.nB, nmax = I.nmax;
            int ks = tbase % STAGES, vs = (tbase + 1) % STAGES;
            uint32_t kph = (tbase / STAGES) & 1, vph = ((tbase + 1) / STAGES) & 1;
            // A launch told to give up (p.give_up) stops at its first wait, before any MMA.
            if (!(ok = (i > 0 || !*abort_flag) && wait_all(b_q_full, i & 1))) break;
            if (nmax > 0) {
                if ((ok = wait_all(b_kv_full(ks), kph))) {
                    tc_fence_after();
                    if (nA > 0) issue_s(0, ks);
                    if (nB > 0) issue_s(1, ks);
                    release(ks);  // K_0: read by both S products above
                }
            }
            // Q_A and Q_B are free for the next item once the item's last S product completes
            auto release_q = [&]() {
                if (leader) mma_commit(b_q_empty);
                __syncwarp();
            };
            if (nmax <= 1) release_q();
            adv(ks, kph);
            for (int j = 0; ok && j < nmax; ++j) {
                const bool more = j + 1 < nmax;
                bool k_ready = false;  // K_{j+1} is waited for only once an S product needs it
                if (!(ok = wait_all(b_kv_full(vs), vph))) break;
                {
                    // Rows past the document's last key (the next document's, the
                    // next batch entry's, or cache slots past seq_len) may hold
                    // anything, NaN included; P is 0 there but 0 * NaN is not, so
                    // the last KV tile's V rows past the end are zeroed first.
                    const int lim = I.Lk - (I.j0 + j) * BN;
                    if (lim < BN) {
                        const uint32_t vb = sKV + vs * C::KV_BYTES;
                        for (int idx = lane; idx < (BN - lim) * NCH * 8; idx += 32) {
                            const int u = idx & 7, rc = idx >> 3, c = rc % NCH, rr = lim + rc / NCH;
                            st_shared_v4(vb + c * BN * 128 + rr * 128 + u * 16, 0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                }
                if (j < nA) {
                    if (!(ok = wait_all(b_p_full(0), (pa + j) & 1))) break;
                    tc_fence_after();
                    issue_pv(0, vs, j > 0);
                    if (j + 1 < nA) {
                        if (!(ok = wait_all(b_kv_full(ks), kph))) break;
                        k_ready = true;
                        tc_fence_after();
                        issue_s(0, ks);
                    }
                }
                if (j < nB) {
                    if (!(ok = wait_all(b_p_full(1), (pb + j) & 1))) break;
                    tc_fence_after();
                    issue_pv(1, vs, j > 0);
                }
                release(vs);  // V_j: its last reader was issued above
                if (j + 1 < nB) {
                    if (!k_ready && !(ok = wait_all(b_kv_full(ks), kph))) break;
                    k_ready = true;
                    tc_fence_after();
                    issue_s(1, ks);
                }
                if (j + 2 == nmax) release_q();  // S_X(nmax - 1) were the item's last S products
                if (more) {
                    if (!k_ready && !(ok = wait_all(b_kv_full(ks), kph))) break;  // keep the phase in step
                    release(ks);  // K_{j+1}: read by the S products issued above
                }
                adv(ks, kph);
                adv(vs, vph);
            }
            tbase += 2 * nmax;
            pa += nA;
            pb += nB;
        }
        // Everything issued above must finish before TMEM is released.
        if (leader) mma_commit(b_drain);
        __syncwarp();
        mbar_wait_drain(b_drain, 0);
      }
      __syncwarp();
      if (split) {  // the three cluster barriers of split_merge
          cluster_sync();
          cluster_sync();
          cluster_sync();
      }
    } else {
        regs_inc<C::REG_SOFTMAX>();
        // ------------------------------------------------------------- softmax
        const int x = warp >> 2;               // 0: tile A, 1: tile B
        const int r = threadIdx.x & 127;       // row within the tile == TMEM lane
        const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t tS = tl + C::TMEM_S + x * BN;
        const uint32_t tO = tl + C::TMEM_O + x * D;
        const float c2 = p.scale_log2;
        uint32_t sdone = 0;  // S_X products of earlier items (phase count of s_full and pv_done)
        int tbase = 0;       // ring index of the item's K_0 (as the producer and MMA warps count)
        bool owe_staged = false;  // (DEFER, thread r == 0) the previous item's last stores
        auto settle_staged = [&]() {
            if (owe_staged) {
                bulk_wait_read0();
                mbar_arrive(b_staged(x));
                owe_staged = false;
            }
        };
        Walk W = walk_here(0xffffffffu);
        for (int i = 0; ok; ++i) {
        const Item I = item_at(i, W);
        if (!I.valid) break;
        const int h = I.h, doc = I.doc, q_start = I.q_start, Lq = I.Lq, Lqu = I.Lqu, Lk = I.Lk, q0 = I.q0,
                  diag = I.diag;
        const int nA = I.nA, nB = I.nB, nmax = I.nmax, j0 = I.j0;
        const int row = q0 + x * TPT + r / gq;  // token within the document
        const int hh = h + r % gq;              // query head of this row
        const int n_kv = x ? nB : nA;
        const int qfirst = q0 + x * TPT;
        // keys [0, row_lim) visible
        const int row_lim = row >= Lqu ? 0 : (p.causal ? min(Lk, row + diag + 1) : Lk);
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < n_kv; ++j) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_s_full(x), (sdone + j) & 1, abort_flag)))) break;
            tc_fence_after();
            const int kbase = (j0 + j) * BN;
            const bool edge =
                (kbase + BN > Lk) || (p.causal && kbase + BN - 1 > qfirst + diag) || qfirst + TPT > Lqu;
            const int lim = row_lim - kbase;  // columns >= lim are masked (edge tiles only)
            uint32_t sr[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
                tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
            tmem_wait_ld();
            if (edge) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
            }
            // row max: three-input max into 4 independent chains (16 deep, 2 values per op)
            float mxp[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) mxp[i] = __uint_as_float(sr[i]);
#pragma unroll
            for (int c = 4; c < BN; c += 2)
                mxp[(c >> 1) & 3] = fmax3(mxp[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            const float mx = fmaxf(fmax3(mxp[0], mxp[1], mxp[2]), mxp[3]);
            const float m_new = fmaxf(m, mx * c2);
            const bool need = m_new > m + kRescaleThreshold;
            const bool warp_need = __any_sync(0xffffffffu, need);
            float alpha = 1.f;
            if (warp_need && m_new > m) {
                alpha = ex2(m - m_new);
                m = m_new;
            }
            l *= alpha;
            // O_X already holds every PV_X(i < j): S_X(j) was issued after them
            if (warp_need && j > 0) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + c * 32, o);
                }
            }
            // P = 2^(S c - m) as bf16 pairs over the first 64 columns of S
            const float msub = (m == -INFINITY) ? 0.f : m;
            const float2 c2x2 = make_float2(c2, c2), negm = make_float2(-msub, -msub);
            float2 rsp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};  // independent partial row sums, in pairs
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 t = __ffma2_rn(
                        make_float2(__uint_as_float(sr[c * 32 + e]), __uint_as_float(sr[c * 32 + e + 1])), c2x2, negm);
                    const float2 pp = make_float2(ex2(t.x), ex2(t.y));
                    rsp[(e >> 1) & 3] = __fadd2_rn(rsp[(e >> 1) & 3], pp);
                    pk[e >> 1] = pack_bf16x2(pp.x, pp.y);
                }
                tmem_st16(tS + c * 16, pk);
            }
            const float2 rr = __fadd2_rn(__fadd2_rn(rsp[0], rsp[1]), __fadd2_rn(rsp[2], rsp[3]));
            l += rr.x + rr.y;
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b_p_full(x));
            if constexpr (DEFER) settle_staged();
        }
        if constexpr (DEFER) settle_staged();  // (an item without KV tiles, or a loop left early)
        ok = __all_sync(0xffffffffu, ok);
        if (ok && n_kv > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(b_pv_done(x), (sdone + n_kv - 1) & 1, abort_flag));
            tc_fence_after();
        }
        sdone += n_kv;
        // ------------------------------------------------------------ epilogue
        if (split) {
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(b_drain, 0, abort_flag));  // all MMAs done
            tc_fence_after();
            split_merge<D>(smem, sKV, tO, x * BM + r, m, l, n_kv > 0, ok, crank, q0, Lq, q_start, h, doc, p);
        } else if (nmax > 0 && qfirst + TPT <= Lq && (x == 1 ? nB >= nA : nA >= nB)) {
            // A tile wholly inside its document leaves through shared memory:
            // its rows are staged in the TMA 128-byte-swizzled box layout
            // (128 rows x 128 bytes per 16 KB box) in a stage of the K/V area
            // and written by tiled TMA stores.  Only a tile that finishes last
            // (or with the other) stages: once PV_X(last) is complete the only
            // MMA that may still read the K/V area is PV_B(last), when tile A
            // finishes with nA == nB: it reads V_{n-1}, whose stage tile A
            // does not use.  A tile with fewer KV tiles than the other (tile A
            // of a causal item, or tile B wholly in the padding of a padded
            // batch) stores directly instead, while the other tile computes on.
            const bool f32 = p.out_f32 != 0;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const int boxes = f32 ? D / 32 : (D + 63) / 64, cols = f32 ? 32 : 64;  // 128-byte boxes per row
            // One K/V stage per tile, NCH boxes at a time: tile B's is V_{n-1}'s
            // (PV_B(last) is complete here), tile A's K_{n-1}'s (every S product
            // is complete once PV_A(last) is; PV_B(last) reads only V_{n-1}).
            // Neither is the next item's K_0 stage, nor those of its next loads
            // but the last two of a ring turn, which wait for these stores.
            const int sk = (tbase + 2 * nmax) % STAGES;
            const uint32_t stage_base = sKV + static_cast<uint32_t>((sk + STAGES - 2 + x) % STAGES) * C::KV_BYTES;
            const int sw = r & 7;
            auto load_scaled = [&](int c, uint32_t (&o)[32]) {
                if (n_kv > 0 && ok) {
                    tmem_ld32(tO + c * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
            };
            for (int b0 = 0; b0 < boxes; b0 += NCH) {
                const int b1 = min(boxes, b0 + NCH);
                if (b0 > 0) named_bar_sync(1 + x, 128);  // the previous boxes' stores have read the stage
                if (f32) {  // 32 columns = one 128-byte box row, 8 units of 16 bytes
#pragma unroll 1
                    for (int b = b0; b < b1; ++b) {
                        uint32_t o[32];
                        load_scaled(b, o);
                        const uint32_t rb = stage_base + static_cast<uint32_t>(b - b0) * (BM * 128) + r * 128;
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            st_shared_v4(rb + ((k ^ sw) << 4), o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                    }
                } else {    // 32 columns = half a box row
#pragma unroll 1
                    for (int c = 2 * b0; c < 2 * b1 && c < D / 32; ++c) {
                        uint32_t o[32];
                        load_scaled(c, o);
                        const uint32_t rb = stage_base + static_cast<uint32_t>((c >> 1) - b0) * (BM * 128) + r * 128;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            st_shared_v4(rb + ((((c & 1) * 4 + k) ^ sw) << 4),
                                         pack_bf16x2(__uint_as_float(o[8 * k]), __uint_as_float(o[8 * k + 1])),
                                         pack_bf16x2(__uint_as_float(o[8 * k + 2]), __uint_as_float(o[8 * k + 3])),
                                         pack_bf16x2(__uint_as_float(o[8 * k + 4]), __uint_as_float(o[8 * k + 5])),
                                         pack_bf16x2(__uint_as_float(o[8 * k + 6]), __uint_as_float(o[8 * k + 7])));
                    }
                }
                fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine
                named_bar_sync(1 + x, 128);
                if (r == 0) {
                    for (int b = b0; b < b1; ++b)
                        tma_store_3d(&tmO, stage_base + static_cast<uint32_t>(b - b0) * (BM * 128), b * cols, h,
                                     q_start + qfirst);
                    bulk_commit();
                    if (DEFER && persist && b1 == boxes)
                        owe_staged = true;  // waited for after the next item's first P
                    else
                        bulk_wait_read0();  // the staging area must outlive the reads
                }
            }
            if (r == 0 && persist && !DEFER) mbar_arrive(b_staged(x));
            if (ok && p.lse) {
                const long long lrow = p.lse_row_global ? (q_start + row) : row;
                p.lse[doc * p.lse_bstride + hh * p.lse_hstride + lrow] =
                    l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
            }
        } else {
        const bool row_valid = ok && row < Lq;
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const long long orow = static_cast<long long>(q_start + row) * p.Hq + hh;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (n_kv > 0 && ok) {
                tmem_ld32(tO + c * 32, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            if (row_valid) {
                if (p.out_f32) {
                    float* dst = reinterpret_cast<float*>(p.out) + orow * D + c * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        st_global_v4(dst + e, __float_as_uint(__uint_as_float(o[e]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 1]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 2]) * inv_l),
                                     __float_as_uint(__uint_as_float(o[e + 3]) * inv_l));
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + orow * D + c * 32;
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
        if (row_valid && p.lse) {
            const long long lrow = p.lse_row_global ? (q_start + row) : row;
            p.lse[doc * p.lse_bstride + hh * p.lse_hstride + lrow] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
        }
        }
        tbase += 2 * nmax;
        }  // items
        if constexpr (DEFER) settle_staged();
    }

    // --------------------------------------------------------------- teardown
    if (!ok) {
        *abort_flag = 1;
        if (p.status) atomicOr(p.status, kDevTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    // A split last wave overlaps the end of the grid before it: it finishes
    // only after that grid, so the stream's later work still follows both.
    if (split) grid_dependency_wait();
}

// ---------------------------------------------------------------- launchers
// D <= 128: two query tiles per CTA; D = 192, 256: one tile (two O
// accumulators of that width do not fit next to the S buffers in TMEM).
using Cfg64 = Prefill2Cfg<64, 10>;
using Cfg96 = Prefill2Cfg<96, 5>;
using Cfg128 = Prefill2Cfg<128, 5>;
using Cfg192 = PrefillCfg<192, 128, 3, 3>;
using Cfg256 = PrefillCfg<256, 128, 5, 2>;

// Sets the dynamic shared-memory limit of `kernel` once per device (one flag
// set per instantiation: the kernels of several configurations share a type).
template <class C, bool PAGED, bool WALK = false, bool DEFER = false, class K>
static cudaError_t set_smem_attr(K kernel, int bytes) {
    static bool done[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

template <class C, bool PAGED, class K>
static cudaError_t launch_kernel(K kernel, int threads, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmO, const PrefillParams& p,
                                 int rows_per_cta, cudaStream_t stream) {
    cudaError_t e = set_smem_attr<C, PAGED>(kernel, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((p.max_seqlen_q + rows_per_cta - 1) / rows_per_cta, p.Hq, p.num_docs);
    kernel<<<grid, threads, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmO, p);
    return cudaGetLastError();
}

// Clusters of `c` CTAs of `kernel` that can be resident at once (cached per
// device and cluster size; 0 if the query fails).
template <class C, class K>
static int resident_clusters(K kernel, int c) {
    static int cache[64][4];
    static bool have[64][4];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int slot = c == 2 ? 0 : c == 4 ? 1 : 2;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev][slot]) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = c;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(c);
        cfg.blockDim = dim3(384);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        cache[dev][slot] = n;
        have[dev][slot] = true;
    }
    return cache[dev][slot];
}

// Launch plan of the two-tile kernel.  Varlen: one launch on a 3D grid
// (tile, head, document).  Dense: a 1D grid of items (tile, head, batch).
// When the last wave of a dense non-causal launch would be less than half
// full, its items go to a second launch in which a cluster of `split` CTAs
// shares each item along the keys and merges the partial results on chip,
// so that the wave lasts about 1/split of an item instead of a whole one.
template <class C, bool PAGED, bool DEFER = false, class K>
static cudaError_t plan_two_tile(K kernel, const PrefillParams& p, int num_sms, PrefillPlan* pl) {
    *pl = PrefillPlan{};
    if (p.cu_q) {
        const int tpt = p.gqa_pack ? 128 / p.group : 128;
        pl->n_items = pl->n_full =
            static_cast<long long>((p.max_seqlen_q + 2 * tpt - 1) / (2 * tpt)) * (p.gqa_pack ? p.Hkv : p.Hq) * p.num_docs;
        pl->launches = pl->n_items > 0 ? 1 : 0;
        // Packed documents whose grid would run more than one wave: one CTA
        // per SM walks the tile-major item list (the walk rescans cu_seqlens
        // per level, so very many documents keep the one-CTA-per-item grid).
        pl->persist = !PAGED && num_sms > 0 && pl->n_items > num_sms && pl->n_items <= 0x7fffffffLL &&
                      p.num_docs <= kWalkMaxDocs;
        return cudaSuccess;
    }
    cudaError_t e = set_smem_attr<C, PAGED, false, DEFER>(kernel, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    pl->tiles = (p.Sq + 255) / 256;
    pl->n_items = static_cast<long long>(pl->tiles) * p.Hq * p.num_docs;
    if (pl->n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
    const int n_kv = (p.Sk + C::BN - 1) / C::BN;
    const int tail = num_sms > 0 ? static_cast<int>(pl->n_items % num_sms) : 0;
    if (!p.causal && tail > 0 && 2 * tail <= num_sms) {
        for (int c = 8; c >= 2 && !pl->split; c >>= 1)
            if (tail * c <= num_sms && n_kv >= 4 * c && resident_clusters<C>(kernel, c) >= tail) pl->split = c;
    }
    pl->n_full = pl->split ? pl->n_items - tail : pl->n_items;
    pl->launches = (pl->n_full > 0 ? 1 : 0) + (pl->split ? 1 : 0);
    // More than one wave (non-causal, so equal items): one CTA per SM walks
    // the full-wave items in turn, so that launch, set-up and the next item's
    // Q and K_0 loads and first S products overlap the current item's work.
    pl->persist = !p.causal && num_sms > 0 && pl->n_full > num_sms;
    return cudaSuccess;
}

template <class C, bool PAGED, bool DEFER = false, class K>
static cudaError_t launch_two_tile(K kernel, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                   const CUtensorMap& tmO, const PrefillParams& p, int num_sms, cudaStream_t stream) {
    PrefillPlan pl;
    cudaError_t e = plan_two_tile<C, PAGED, DEFER>(kernel, p, num_sms, &pl);
    if (e != cudaSuccess) return e;
    e = set_smem_attr<C, PAGED, false, DEFER>(kernel, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PrefillParams q = p;
    q.split = 0;
    q.item_base = 0;
    if (p.cu_q && pl.persist) {  // the walk is its own instantiation (non-paged only)
        if (PAGED) return cudaErrorInvalidValue;
        // (packed documents give many items of few KV tiles: the DEFER form)
        auto walk = fmha2_fwd_sm103a<C, false, true, true>;
        if ((e = set_smem_attr<C, false, true, true>(walk, C::SMEM_BYTES)) != cudaSuccess) return e;
        q.linear = 2;
        q.persist = 1;
        walk<<<static_cast<unsigned>(num_sms), 384, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmO, q);
        return cudaGetLastError();
    }
    if (p.cu_q) {
        q.linear = 0;
        const int tpt = p.gqa_pack ? 128 / p.group : 128;  // tokens per tile
        dim3 grid((p.max_seqlen_q + 2 * tpt - 1) / (2 * tpt), p.gqa_pack ? p.Hkv : p.Hq, p.num_docs);
        kernel<<<grid, 384, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmO, q);
        return cudaGetLastError();
    }
    q.linear = 1;
    q.tiles = pl.tiles;
    if (pl.n_full > 0) {
        q.persist = pl.persist;
        q.item_end = static_cast<int>(pl.n_full);
        const long long grid = pl.persist ? std::min<long long>(pl.n_full, num_sms) : pl.n_full;
        kernel<<<static_cast<unsigned>(grid), 384, C::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, tmO, q);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        q.persist = 0;
    }
    if (pl.split) {
        q.item_base = static_cast<int>(pl.n_full);
        q.split = pl.split;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = pl.split;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        // behind the full-wave launch: start as its CTAs finish
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(static_cast<unsigned>((pl.n_items - pl.n_full) * pl.split));
        cfg.blockDim = dim3(384);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = at;
        cfg.numAttrs = pl.n_full > 0 ? 2 : 1;
        e = cudaLaunchKernelEx(&cfg, kernel, tmQ, tmK, tmV, tmO, q);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// The paged mode (K/V through block_table) is a separate instantiation, so
// that the dense and varlen kernels carry none of its code.
template <class C>
static cudaError_t two_tile(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmO, const PrefillParams& p, int num_sms, cudaStream_t stream) {
    if (p.block_table)
        return launch_two_tile<C, true>(fmha2_fwd_sm103a<C, true, false>, tmQ, tmK, tmV, tmO, p, num_sms, stream);
    // dense launches of at most 8 KV tiles per item spend much of an item in
    // its epilogue: the instantiation that defers the staged stores' wait
    if (!p.cu_q && !p.causal && (p.Sk + C::BN - 1) / C::BN <= 8)
        return launch_two_tile<C, false, true>(fmha2_fwd_sm103a<C, false, false, true>, tmQ, tmK, tmV, tmO, p, num_sms,
                                               stream);
    return launch_two_tile<C, false>(fmha2_fwd_sm103a<C, false, false>, tmQ, tmK, tmV, tmO, p, num_sms, stream);
}

template <class C>
static cudaError_t one_tile(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmO, const PrefillParams& p, cudaStream_t stream) {
    return p.block_table ? launch_kernel<C, true>(fmha_fwd_sm103a<C, true>, 192, tmQ, tmK, tmV, tmO, p, 128, stream)
                         : launch_kernel<C, false>(fmha_fwd_sm103a<C, false>, 192, tmQ, tmK, tmV, tmO, p, 128, stream);
}

template <class C>
static cudaError_t plan_for(const PrefillParams& p, int num_sms, PrefillPlan* pl) {
    return p.block_table ? plan_two_tile<C, true>(fmha2_fwd_sm103a<C, true, false>, p, num_sms, pl)
                         : plan_two_tile<C, false>(fmha2_fwd_sm103a<C, false, false>, p, num_sms, pl);
}

int prefill_block_n(int D) { return (D == 64 || D == 96 || D == 128 || D == 192 || D == 256) ? 128 : 0; }
int prefill_v_box_rows(int D) { return D == 256 ? Cfg256::VR : D == 192 ? Cfg192::VR : prefill_block_n(D); }

cudaError_t launch_prefill(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmO, const PrefillParams& p, int num_sms, cudaStream_t stream) {
    switch (D) {
        case 64: return two_tile<Cfg64>(tmQ, tmK, tmV, tmO, p, num_sms, stream);
        case 96: return two_tile<Cfg96>(tmQ, tmK, tmV, tmO, p, num_sms, stream);
        case 128: return two_tile<Cfg128>(tmQ, tmK, tmV, tmO, p, num_sms, stream);
        case 192: return one_tile<Cfg192>(tmQ, tmK, tmV, tmO, p, stream);
        case 256: return one_tile<Cfg256>(tmQ, tmK, tmV, tmO, p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t prefill_plan(int D, const PrefillParams& p, int num_sms, PrefillPlan* pl) {
    switch (D) {
        case 64: return plan_for<Cfg64>(p, num_sms, pl);
        case 96: return plan_for<Cfg96>(p, num_sms, pl);
        case 128: return plan_for<Cfg128>(p, num_sms, pl);
        case 192:
        case 256: {
            *pl = PrefillPlan{};
            pl->n_items = pl->n_full = static_cast<long long>((p.max_seqlen_q + 127) / 128) * p.Hq * p.num_docs;
            pl->launches = pl->n_items > 0 ? 1 : 0;
            return cudaSuccess;
        }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbattn
