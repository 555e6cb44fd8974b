"""The benchmarks' denominators and inputs, checked on the CPU: every FLOP or
byte count a bench line divides by is recounted here from the oracle's
visibility rule or from the tensors themselves."""

import numpy as np
import torch

import oracle
import workloads


def _pairs(lq, lk, causal):
    return int(oracle.visible_mask(lq, lk, causal).sum())


def test_dense_and_varlen_flops_count_the_visible_pairs():
    for w in (workloads.Dense("a", 2, 300, 170, 4, 2, 64, True, seed=0),
              workloads.Dense("b", 1, 100, 300, 2, 2, 128, False, seed=0)):
        assert w.flops() == 4.0 * w.D * w.B * w.Hq * _pairs(w.Sq, w.Sk, w.causal)
    v = workloads.Varlen("c", [5, 300, 17], [40, 300, 3], 4, 2, 64, True, seed=0)
    assert v.flops() == 4.0 * 64 * 4 * sum(_pairs(a, b, True) for a, b in zip(v.lens_q, v.lens_k))


def test_paged_prefill_flops_count_the_visible_pairs():
    w = workloads.PagedPrefill("d", [300, 1, 1000, 50], [16, 1, 200, 80], 8, 2, 128, seed=1)
    assert w.flops() == 4.0 * 128 * 8 * sum(_pairs(q, k, True) for q, k in zip(w.q_lens, w.seq_lens))
    assert workloads.chunked_prefill().q_lens == [512] * 16
    assert workloads.spec_decode().seq_lens == workloads.paged_decode().seq_lens  # same contexts as the decode


def test_masked_flops_count_the_kept_pairs():
    w = workloads.Masked("e", [40, 17], 64, 2, 2, 32, True, seed=2)
    q, k, v, mask = w.make()
    assert mask.sum(dim=1).tolist() == [40, 17] and mask.shape == (2, 64)
    assert w.flops() == 4.0 * 32 * 2 * sum(_pairs(n, n, True) for n in w.lens)
    assert workloads.masked_dit().flops() == 4.0 * 128 * 24 * (4096 ** 2 + 3072 ** 2)


def test_cache_write_slots_and_bytes():
    w = workloads.CacheWrite("f", [5, 130, 256, 1], 2, 64, seed=3)
    k, v, slots, shape = w.make()
    assert shape == (2, w.num_blocks, 128, 2, 64) and w.num_blocks == 1 + 2 + 2 + 1
    s = slots.tolist()
    assert len(set(s)) == len(s) == w.tokens and min(s) >= 0 and max(s) < w.num_blocks * 128
    at = 0
    for n in w.lens:  # a document's tokens fill its blocks in order
        blocks = [x // 128 for x in s[at:at + n]]
        offs = [x % 128 for x in s[at:at + n]]
        assert offs == [t % 128 for t in range(n)]
        assert all(blocks[t] == blocks[t - t % 128] for t in range(n))
        at += n
    assert w.algorithmic_bytes() == 2 * (k.numel() + v.numel()) * 2 + 4 * w.tokens


def test_paged_decode_bytes_count_every_context_token_once():
    w = workloads.Paged("g", [1, 129, 300], 8, 2, 64, seed=4)
    q, cache, bt, sl = w.make()
    kv = 2 * sum(w.seq_lens) * 2 * 64 * 2
    blocks = sum(-(-n // 128) for n in w.seq_lens)
    assert w.algorithmic_bytes() == kv + 4 * blocks + 4 * 3 + q.numel() * 2 + 3 * 8 * 64 * 4 + 3 * 8 * 4
    used = bt[bt >= 0]
    assert len(set(used.tolist())) == blocks  # every physical block used once


def test_generators_are_seeded_and_bf16():
    a = workloads.tiny_varlen().make()
    b = workloads.tiny_varlen().make()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert a[0].dtype == torch.bfloat16 and np.isfinite(a[0].float().numpy()).all()


def test_vsa_kept_pairs_count_the_block_map():
    """The block-sparse bench divides by 4 D x the query-key pairs its lists
    keep; recounted here from the oracle's block map itself."""
    import bench
    from _helpers import vsa_lists_from_map

    prefix, video, topk = [100, 37], (5, 9, 10), 5
    blocks, npre = oracle.vsa_blocks(prefix, video)
    n = sum(prefix) + int(np.prod(video))
    g = torch.Generator().manual_seed(7)
    q, k = torch.randn(n, 3, 16, generator=g), torch.randn(n, 3, 16, generator=g)
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk, 0.25)
    sizes = [len(b) for b in blocks]
    kl, kn = vsa_lists_from_map(bm, sizes, npre, topk)
    expect = sum(sizes[i] * sum(sizes[j] for j in np.nonzero(bm[h, i])[0])
                 for h in range(3) for i in range(len(blocks)))
    assert bench.vsa_kept_pairs(kl, kn, len(blocks), npre, topk, sizes) == expect
    w = workloads.vsa_video()
    assert w.tokens == 512 + 21 * 45 * 80 and w.topk == 64
