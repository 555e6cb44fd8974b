// vsa_layout.cpp -- token layout of block-sparse video attention (host code).
//
// Operation: vllm-omni fastvideo_vsa.py, _get_h3_tile_metadata -- the
// sequence is a prefix (segments cut into chunks of `block` tokens) followed
// by a (T, H, W) video latent grid in T, H, W order, cut into boxes of
// tile_t x tile_h x tile_w tokens taken in T, H, W order (boxes at the far
// edges of the grid are smaller).  The layout is a pure function of the
// sizes, so it is computed once on the host, as on the page.
#include <stdint.h>

#include "../../include/gbattn.h"

namespace {

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Calls blk(first token slot, count) once per block in layout order and
// tok(token) once per token, in order, after its block's blk call.
template <class Blk, class Tok>
void walk_layout(const int32_t* prefix_segments, int num_segments, long long T, long long H, long long W, int tile_t,
                 int tile_h, int tile_w, int block, Blk blk, Tok tok) {
    long long base = 0;
    for (int i = 0; i < num_segments; ++i) {
        for (long long c0 = 0; c0 < prefix_segments[i]; c0 += block) {
            const long long c1 = c0 + block < prefix_segments[i] ? c0 + block : prefix_segments[i];
            blk(c1 - c0);
            for (long long t = c0; t < c1; ++t) tok(base + t);
        }
        base += prefix_segments[i];
    }
    for (long long i = 0; i < ceil_div(T, tile_t); ++i)
        for (long long j = 0; j < ceil_div(H, tile_h); ++j)
            for (long long k = 0; k < ceil_div(W, tile_w); ++k) {
                const long long t1 = (i + 1) * tile_t < T ? (i + 1) * tile_t : T;
                const long long h1 = (j + 1) * tile_h < H ? (j + 1) * tile_h : H;
                const long long w1 = (k + 1) * tile_w < W ? (k + 1) * tile_w : W;
                blk((t1 - i * tile_t) * (h1 - j * tile_h) * (w1 - k * tile_w));
                for (long long t = i * tile_t; t < t1; ++t)
                    for (long long h = j * tile_h; h < h1; ++h)
                        for (long long w = k * tile_w; w < w1; ++w) tok(base + (t * H + h) * W + w);
            }
}

// Validates the geometry and counts blocks; GBATTN_OK or an error status.
gbattn_status layout_counts(const int32_t* prefix_segments, int num_segments, int T, int H, int W, int tile_t,
                            int tile_h, int tile_w, int block, long long* nb_out, long long* npre_out) {
    if (num_segments < 0 || (num_segments > 0 && !prefix_segments) || T < 0 || H < 0 || W < 0 || tile_t <= 0 ||
        tile_h <= 0 || tile_w <= 0 || block <= 0)
        return GBATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(tile_t) * tile_h * tile_w > block) return GBATTN_ERR_INVALID_ARG;  // a box fits a block
    long long prefix = 0, nb = 0;
    for (int i = 0; i < num_segments; ++i) {
        if (prefix_segments[i] < 0) return GBATTN_ERR_INVALID_ARG;
        prefix += prefix_segments[i];
        nb += ceil_div(prefix_segments[i], block);
    }
    *npre_out = nb;
    nb += ceil_div(T, tile_t) * ceil_div(H, tile_h) * ceil_div(W, tile_w);
    const long long total = prefix + static_cast<long long>(T) * H * W;
    if (total > 0x7fffffffLL || nb > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    *nb_out = nb;
    return GBATTN_OK;
}

}  // namespace

extern "C" {

gbattn_status attn_vsa_layout(const int32_t* prefix_segments, int num_segments, int T, int H, int W, int tile_t,
                              int tile_h, int tile_w, int block, int32_t* order, int32_t* block_start,
                              int* num_blocks, int* num_prefix_blocks) {
    if (!num_blocks || !num_prefix_blocks) return GBATTN_ERR_INVALID_ARG;
    long long nb = 0, npre = 0;
    const gbattn_status s =
        layout_counts(prefix_segments, num_segments, T, H, W, tile_t, tile_h, tile_w, block, &nb, &npre);
    if (s != GBATTN_OK) return s;
    *num_blocks = static_cast<int>(nb);
    *num_prefix_blocks = static_cast<int>(npre);
    if (!order || !block_start) return GBATTN_OK;  // sizes only
    long long at = 0, b = 0;
    walk_layout(
        prefix_segments, num_segments, T, H, W, tile_t, tile_h, tile_w, block,
        [&](long long) { block_start[b++] = static_cast<int32_t>(at); },
        [&](long long tok) { order[at++] = static_cast<int32_t>(tok); });
    block_start[b] = static_cast<int32_t>(at);
    return GBATTN_OK;
}

gbattn_status attn_vsa_tile_map(const int32_t* prefix_segments, int num_segments, int T, int H, int W, int tile_t,
                                int tile_h, int tile_w, int32_t* tile_index, int32_t* block_sizes, int* num_blocks,
                                int* num_prefix_blocks) {
    if (!num_blocks || !num_prefix_blocks) return GBATTN_ERR_INVALID_ARG;
    long long nb = 0, npre = 0;
    const gbattn_status s =
        layout_counts(prefix_segments, num_segments, T, H, W, tile_t, tile_h, tile_w, 64, &nb, &npre);
    if (s != GBATTN_OK) return s;
    if ((nb + 1) / 2 * 128 > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;  // tiled rows fit int32
    *num_blocks = static_cast<int>(nb);
    *num_prefix_blocks = static_cast<int>(npre);
    if (!tile_index || !block_sizes) return GBATTN_OK;  // sizes only
    const long long rows = (nb + (nb & 1)) * 64;
    for (long long r = 0; r < rows; ++r) tile_index[r] = -1;
    long long b = -1, r = 0;
    walk_layout(
        prefix_segments, num_segments, T, H, W, tile_t, tile_h, tile_w, 64,
        [&](long long n) {
            block_sizes[++b] = static_cast<int32_t>(n);
            r = 0;
        },
        [&](long long tok) { tile_index[b * 64 + r++] = static_cast<int32_t>(tok); });
    return GBATTN_OK;
}

}  // extern "C"
