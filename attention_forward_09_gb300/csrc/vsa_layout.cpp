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

}  // namespace

extern "C" {

gbattn_status attn_vsa_layout(const int32_t* prefix_segments, int num_segments, int T, int H, int W, int tile_t,
                              int tile_h, int tile_w, int block, int32_t* order, int32_t* block_start,
                              int* num_blocks, int* num_prefix_blocks) {
    if (num_segments < 0 || (num_segments > 0 && !prefix_segments) || T < 0 || H < 0 || W < 0 || tile_t <= 0 ||
        tile_h <= 0 || tile_w <= 0 || block <= 0 || !num_blocks || !num_prefix_blocks)
        return GBATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(tile_t) * tile_h * tile_w > block) return GBATTN_ERR_INVALID_ARG;  // a box fits a block
    long long prefix = 0, nb = 0;
    for (int i = 0; i < num_segments; ++i) {
        if (prefix_segments[i] < 0) return GBATTN_ERR_INVALID_ARG;
        prefix += prefix_segments[i];
        nb += ceil_div(prefix_segments[i], block);
    }
    const long long npre = nb;
    const long long nt = ceil_div(T, tile_t), nh = ceil_div(H, tile_h), nw = ceil_div(W, tile_w);
    nb += nt * nh * nw;
    const long long total = prefix + static_cast<long long>(T) * H * W;
    if (total > 0x7fffffffLL || nb > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    *num_blocks = static_cast<int>(nb);
    *num_prefix_blocks = static_cast<int>(npre);
    if (!order || !block_start) return GBATTN_OK;  // sizes only
    long long at = 0, b = 0, base = 0;
    for (int i = 0; i < num_segments; ++i) {
        for (long long c0 = 0; c0 < prefix_segments[i]; c0 += block) {
            block_start[b++] = static_cast<int32_t>(at);
            const long long c1 = c0 + block < prefix_segments[i] ? c0 + block : prefix_segments[i];
            for (long long t = c0; t < c1; ++t) order[at++] = static_cast<int32_t>(base + t);
        }
        base += prefix_segments[i];
    }
    for (long long i = 0; i < nt; ++i)
        for (long long j = 0; j < nh; ++j)
            for (long long k = 0; k < nw; ++k) {
                block_start[b++] = static_cast<int32_t>(at);
                for (long long t = i * tile_t; t < T && t < (i + 1) * tile_t; ++t)
                    for (long long h = j * tile_h; h < H && h < (j + 1) * tile_h; ++h)
                        for (long long w = k * tile_w; w < W && w < (k + 1) * tile_w; ++w)
                            order[at++] = static_cast<int32_t>(prefix + (t * H + h) * W + w);
            }
    block_start[b] = static_cast<int32_t>(at);
    return GBATTN_OK;
}

}  // extern "C"
