"""Pins of the float64 oracle against facts fixed outside it.

Each pin is chosen so that a plausible slip in the oracle fails it: a wrong
mask offset (causal pins, q = 0 closed form), a wrong GQA head map (one-hot
routing), K and V indices mixed up (joint vs V-only permutation), a dropped
normalisation (V = const, weights sum to one), a wrong LSE (hand-worked
values, Decimal brute force, scipy's logsumexp), broken document or block
indexing (pack vs separate runs, paged scatter vs contiguous).
"""

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _rand(*shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- hand-worked

def _golden_cases():
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked(case):
    q = np.array(case["q_full"], dtype=np.float64)
    k = np.array(case["k"], dtype=np.float64)
    v = np.array(case["v"], dtype=np.float64)
    out, lse = oracle.attention_single(q, k, v, case["scale"], case["causal"])
    want_lse = np.array([[float(x) for x in row] for row in case["lse"]])
    np.testing.assert_allclose(out, np.array(case["out"]), rtol=0, atol=1e-13)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], want_lse[fin], rtol=0, atol=1e-13)
    assert np.all(lse[~fin] == -np.inf)


# --------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", [(5, 5), (3, 7), (7, 3), (1, 9)])
def test_zero_query_is_mean_of_visible_values(causal, lq, lk):
    """q = 0 makes every visible score 0: out = mean of the visible V rows and
    lse = ln(number visible); the bottom-right rule gives row i
    clip(i + 1 + lk - lq, 0, lk) visible keys."""
    hq, hkv, d = 6, 3, 4
    q = np.zeros((lq, hq, d))
    k, v = _rand(lk, hkv, d), _rand(lk, hkv, d)
    out, lse = oracle.attention_single(q, k, v, 0.3, causal)
    for i in range(lq):
        n = lk if not causal else min(lk, max(0, i + 1 + lk - lq))
        for h in range(hq):
            kv = h // (hq // hkv)
            if n == 0:
                assert np.all(out[i, h] == 0) and lse[h, i] == -np.inf
            else:
                np.testing.assert_allclose(out[i, h], v[:n, kv].mean(axis=0), atol=1e-13)
                assert abs(lse[h, i] - math.log(n)) < 1e-13


def test_single_key_returns_its_value_row():
    d = 16
    q, k, v = _rand(4, 2, d), _rand(1, 1, d), _rand(1, 1, d)
    out, lse = oracle.attention_single(q, k, v, 0.25, False)
    for h in range(2):
        np.testing.assert_array_equal(out[:, h], np.repeat(v[:, 0], 4, axis=0))
        np.testing.assert_allclose(lse[h], 0.25 * q[:, h] @ k[0, 0], atol=1e-13)


def test_identical_value_rows_and_constant_values():
    lq, lk, d = 6, 11, 8
    q, k = _rand(lq, 2, d), _rand(lk, 2, d)
    row = _rand(d)
    v = np.broadcast_to(row, (lk, 2, d)).copy()
    out, _ = oracle.attention_single(q, k, v, 0.5, True)
    np.testing.assert_allclose(out, np.broadcast_to(row, out.shape), atol=1e-13)
    out1, _ = oracle.attention_single(q, k, np.ones((lk, 2, d)), 0.5, False)
    np.testing.assert_allclose(out1, 1.0, atol=1e-14)


def test_one_hot_routing_pins_gqa_head_map():
    """Query head h puts all its weight on key h; out[h] must then be V row h
    of KV head h // (Hq/Hkv) -- not h % Hkv, not another key."""
    hq, hkv, d = 8, 2, 8
    q = np.zeros((1, hq, d))
    for h in range(hq):
        q[0, h, h] = 60.0
    k = np.zeros((d, hkv, d))
    for j in range(d):
        k[j, :, j] = 1.0
    v = _rand(d, hkv, d)
    out, _ = oracle.attention_single(q, k, v, 1.0, False)
    for h in range(hq):
        np.testing.assert_allclose(out[0, h], v[h, h // (hq // hkv)], atol=1e-20 + 1e-12)
        assert not np.allclose(out[0, h], v[h, h % hkv]) or h // 4 == h % 2


def test_weights_sum_to_one_and_vanish_where_masked():
    lq, lk, d = 9, 13, 5
    q, k = _rand(lq, 4, d), _rand(lk, 2, d)
    for causal in (False, True):
        for h in range(4):
            w = oracle.softmax_weights(q, k, 0.7, causal, h)
            assert np.all(w >= 0)
            np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
            if causal:
                vis = oracle.visible_mask(lq, lk, True)
                assert np.all(w[~vis] == 0)


def test_permutation_invariance_and_value_sensitivity():
    lq, lk, d = 4, 10, 6
    q, k, v = _rand(lq, 1, d), _rand(lk, 1, d), _rand(lk, 1, d)
    perm = rng.permutation(lk)
    out, lse = oracle.attention_single(q, k, v, 0.4, False)
    out_p, lse_p = oracle.attention_single(q, k[perm], v[perm], 0.4, False)
    np.testing.assert_allclose(out_p, out, atol=1e-13)
    np.testing.assert_allclose(lse_p, lse, atol=1e-13)
    out_v, _ = oracle.attention_single(q, k, v[perm], 0.4, False)
    assert np.max(np.abs(out_v - out)) > 1e-3


def test_affine_in_values():
    lq, lk, d = 5, 7, 4
    q, k, v = _rand(lq, 2, d), _rand(lk, 2, d), _rand(lk, 2, d)
    c = _rand(d)
    out, _ = oracle.attention_single(q, k, v, 0.5, True)
    out2, _ = oracle.attention_single(q, k, 3.0 * v + c, 0.5, True)
    np.testing.assert_allclose(out2, 3.0 * out + c, atol=1e-12)


# ------------------------------------------------- brute force / library pins

def _decimal_attention(q, k, v, scale, causal):
    """Direct sum of exponentials at 50 digits (no max subtraction)."""
    getcontext().prec = 50
    lq, lk = len(q), len(k)
    out, lse = [], []
    for i in range(lq):
        w = []
        for j in range(lk):
            if causal and j > i + (lk - lq):
                continue
            s = Decimal(scale) * sum(Decimal(a) * Decimal(b) for a, b in zip(q[i], k[j]))
            w.append((j, s.exp()))
        z = sum(x for _, x in w)
        out.append([float(sum(x * Decimal(v[j][c]) for j, x in w) / z) for c in range(len(v[0]))])
        lse.append(float(z.ln()))
    return np.array(out), np.array(lse)


@pytest.mark.parametrize("causal", [False, True])
def test_decimal_brute_force_tiny(causal):
    lq, lk, d = 4, 6, 3
    q, k, v = _rand(lq, 1, d) * 2, _rand(lk, 1, d) * 2, _rand(lk, 1, d)
    out, lse = oracle.attention_single(q, k, v, 0.9, causal)
    bo, bl = _decimal_attention(q[:, 0].tolist(), k[:, 0].tolist(), v[:, 0].tolist(), 0.9, causal)
    np.testing.assert_allclose(out[:, 0], bo, atol=1e-12)
    np.testing.assert_allclose(lse[0], bl, atol=1e-12)


def test_lse_matches_scipy_logsumexp():
    scipy_special = pytest.importorskip("scipy.special")
    lq, lk, d = 7, 12, 8
    q, k = _rand(lq, 1, d) * 3, _rand(lk, 1, d)
    _, lse = oracle.attention_single(q, k, _rand(lk, 1, d), 0.35, True)
    for i in range(lq):
        n = i + 1 + lk - lq
        scores = [0.35 * float(np.dot(q[i, 0], k[j, 0])) for j in range(n)]
        assert abs(lse[0, i] - scipy_special.logsumexp(scores)) < 1e-12


# ------------------------------------------------------------ mask identities

def test_causal_last_row_equals_full_single_query():
    lq, lk, d = 6, 9, 8
    q, k, v = _rand(lq, 2, d), _rand(lk, 2, d), _rand(lk, 2, d)
    out_c, lse_c = oracle.attention_single(q, k, v, 0.3, True)
    out_1, lse_1 = oracle.attention_single(q[-1:], k, v, 0.3, False)
    np.testing.assert_allclose(out_c[-1], out_1[0], atol=1e-13)
    np.testing.assert_allclose(lse_c[:, -1], lse_1[:, 0], atol=1e-13)


def test_causal_square_row_is_prefix_attention():
    l, d = 8, 4
    q, k, v = _rand(l, 1, d), _rand(l, 1, d), _rand(l, 1, d)
    out, lse = oracle.attention_single(q, k, v, 0.6, True)
    for i in range(l):
        o, s = oracle.attention_single(q[i:i + 1], k[:i + 1], v[:i + 1], 0.6, False)
        np.testing.assert_allclose(out[i], o[0], atol=1e-13)
        assert abs(lse[0, i] - s[0, 0]) < 1e-13


def test_fully_masked_rows_and_empty_keys():
    q, k, v = _rand(5, 2, 4), _rand(2, 2, 4), _rand(2, 2, 4)
    out, lse = oracle.attention_single(q, k, v, 0.5, True)  # rows 0..2 see nothing
    assert np.all(out[:3] == 0) and np.all(lse[:, :3] == -np.inf)
    assert np.all(np.isfinite(lse[:, 3:]))
    out0, lse0 = oracle.attention_single(q, k[:0], v[:0], 0.5, False)
    assert np.all(out0 == 0) and np.all(lse0 == -np.inf)


def test_power_of_two_prescale_is_exact():
    """Laser-attention prescale (flash_attn.py, FlashAttentionImpl.
    _forward_prefix_kv_slice_npu): q, k, v divided by s = 2 with the scale
    multiplied by s^2, output multiplied back by s, is the same attention."""
    q, k, v = _rand(7, 2, 8), _rand(9, 2, 8), _rand(9, 2, 8)
    out, lse = oracle.attention_single(q, k, v, 0.125, True)
    out2, lse2 = oracle.attention_single(q / 2, k / 2, v / 2, 0.5, True)
    np.testing.assert_array_equal(out2 * 2, out)
    np.testing.assert_array_equal(lse2, lse)


# ------------------------------------------------------ varlen / dense / paged

def test_dense_equals_varlen_with_arange_cu_seqlens():
    """flash_attn.py, FlashAttentionImpl._flash_varlen_wrapper: a dense batch
    is the varlen call with cu_seqlens = arange(0, (B+1)*L, L)."""
    b, sq, sk, hq, hkv, d = 3, 5, 7, 4, 2, 8
    q, k, v = _rand(b, sq, hq, d), _rand(b, sk, hkv, d), _rand(b, sk, hkv, d)
    for causal in (False, True):
        out, lse = oracle.attention_dense(q, k, v, 0.3, causal)
        cq, ck = np.arange(0, (b + 1) * sq, sq), np.arange(0, (b + 1) * sk, sk)
        out_v, lse_v = oracle.attention_varlen(
            q.reshape(b * sq, hq, d), k.reshape(b * sk, hkv, d), v.reshape(b * sk, hkv, d), cq, ck, 0.3, causal)
        np.testing.assert_array_equal(out_v.reshape(out.shape), out)
        np.testing.assert_array_equal(lse_v.reshape(hq, b, sq).transpose(1, 0, 2), lse)


def test_varlen_pack_equals_documents_run_alone():
    lens_q, lens_k = [3, 0, 7, 1], [4, 2, 7, 5]
    hq, hkv, d = 4, 1, 8
    q, k, v = _rand(sum(lens_q), hq, d), _rand(sum(lens_k), hkv, d), _rand(sum(lens_k), hkv, d)
    cq, ck = np.cumsum([0] + lens_q), np.cumsum([0] + lens_k)
    for causal in (False, True):
        out, lse = oracle.attention_varlen(q, k, v, cq, ck, 0.4, causal)
        for n in range(len(lens_q)):
            o, s = oracle.attention_single(q[cq[n]:cq[n + 1]], k[ck[n]:ck[n + 1]], v[ck[n]:ck[n + 1]], 0.4, causal)
            np.testing.assert_array_equal(out[cq[n]:cq[n + 1]], o)
            np.testing.assert_array_equal(lse[:, cq[n]:cq[n + 1]], s)
        # a mistake that lets documents see each other changes the answer
        o_all, _ = oracle.attention_single(q, k, v, 0.4, False)
        assert np.max(np.abs(o_all - out)) > 1e-3


def test_varlen_rejects_bad_cu_seqlens():
    q, k = _rand(4, 1, 2), _rand(4, 1, 2)
    with pytest.raises(ValueError):
        oracle.attention_varlen(q, k, k, [0, 3, 2, 4], [0, 1, 2, 4], 1.0, False)
    with pytest.raises(ValueError):
        oracle.attention_varlen(q, k, k, [0, 4], [0, 3], 1.0, False)


def _scatter_to_pages(ks, vs, nb, bs, seed):
    """Build a paged cache by writing each token to slot block*bs + offset
    through a randomly permuted block table (the inverse of the gather)."""
    r = np.random.default_rng(seed)
    hkv, d = ks[0].shape[1:]
    cache = np.full((2, nb, bs, hkv, d), np.nan)
    perm = r.permutation(nb)
    maxb = max(-(-len(x) // bs) for x in ks)
    bt = np.full((len(ks), maxb), -1)
    at = 0
    for s, (kk, vv) in enumerate(zip(ks, vs)):
        nblk = -(-len(kk) // bs)
        bt[s, :nblk] = perm[at:at + nblk]
        at += nblk
        for t in range(len(kk)):
            slot = bt[s, t // bs] * bs + t % bs
            cache[0].reshape(nb * bs, hkv, d)[slot] = kk[t]
            cache[1].reshape(nb * bs, hkv, d)[slot] = vv[t]
    return cache, bt


def test_paged_equals_contiguous_and_ignores_unused_slots():
    bs, hq, hkv, d = 4, 4, 2, 8
    lens = [5, 1, 8, 11]
    ks = [_rand(n, hkv, d) for n in lens]
    vs = [_rand(n, hkv, d) for n in lens]
    nb = sum(-(-n // bs) for n in lens) + 3
    q = _rand(len(lens), hq, d)
    outs = []
    for seed in (0, 1):
        cache, bt = _scatter_to_pages(ks, vs, nb, bs, seed)
        cache = np.nan_to_num(cache, nan=0.0) + np.where(np.isnan(cache), 1e6, 0.0)  # poison unused slots
        out, lse = oracle.attention_paged(q, cache, bt, lens, 0.3)
        for s in range(len(lens)):
            o, l = oracle.attention_single(q[s:s + 1], ks[s], vs[s], 0.3, False)
            np.testing.assert_array_equal(out[s], o[0])
            np.testing.assert_array_equal(lse[s], l[:, 0])
        outs.append(out)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_paged_gather_rejects_out_of_range_block():
    cache = np.zeros((2, 2, 4, 1, 2))
    with pytest.raises(ValueError):
        oracle.paged_gather(cache, np.array([[0, 5]]), [6])


# ----------------------------------------------------------------- workloads

def test_workload_shapes_and_index_structures():
    w3 = workloads.varlen_causal_gqa()
    assert len(w3.lens_q) == 8 and sum(w3.lens_q) <= 32768
    assert all(512 <= n <= 8192 for n in w3.lens_q)
    w4 = workloads.paged_decode()
    assert len(w4.seq_lens) == 64 and all(1024 <= n <= 32768 for n in w4.seq_lens)
    bt = w4.block_table()
    used = [int(b) for s, n in enumerate(w4.seq_lens) for b in bt[s, :-(-n // 128)]]
    assert sorted(used) == list(range(w4.num_blocks))  # every physical block used exactly once
    assert all(int(x) == -1 for s, n in enumerate(w4.seq_lens) for x in bt[s, -(-n // 128):])
    w1 = workloads.tiny_varlen()
    q, k, v, cq, ck = w1.make()
    assert q.shape == (128, 4, 64) and cq.tolist() == [0, 37, 128]
    assert abs(w1.flops() - 4 * 64 * 4 * (37 ** 2 + 91 ** 2)) < 1
    assert abs(workloads.dit_self().flops() - 412.3e9) / 412.3e9 < 1e-3


# ------------------------------------------------------------- KV cache write

def test_kv_cache_write_pages_example():
    """slot_mapping [35, 2, 17] with blocks of 16 (the AscendMetadata comment)."""
    g = json.load(open(os.path.join(GOLDEN, "slot_mapping_example.json")))
    bs, slots = g["block_size"], g["slot_mapping"]
    cache = torch.zeros(2, 4, bs, 1, 32, dtype=torch.bfloat16)
    k = torch.arange(1, 4, dtype=torch.float32).view(3, 1, 1).expand(3, 1, 32).to(torch.bfloat16)
    new = oracle.kv_cache_write(k, -k, torch.tensor(slots), cache)
    for t, (b, o) in enumerate(g["block_offset"]):
        assert torch.equal(new[0, b, o], k[t]) and torch.equal(new[1, b, o], -k[t])
    assert int((new != 0).any(dim=-1).sum()) == 2 * len(slots)  # nothing else written
    assert torch.equal(cache, torch.zeros_like(cache))          # the input is left alone


def test_kv_cache_write_then_paged_gather_is_identity():
    """Writing every token of every sequence at block_table[s, t // bs] * bs + t % bs
    and reading the cache back through paged_gather returns the tokens bit for bit."""
    gen = torch.Generator().manual_seed(5)
    lens, bs, hkv, d = [5, 33, 16, 1], 16, 2, 32
    nb = sum(-(-n // bs) for n in lens) + 3
    perm = torch.randperm(nb, generator=gen)
    bt = torch.full((len(lens), 4), -1, dtype=torch.int32)
    at = 0
    for s, n in enumerate(lens):
        m = -(-n // bs)
        bt[s, :m] = perm[at:at + m]
        at += m
    k = torch.randn(sum(lens), hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(sum(lens), hkv, d, generator=gen).to(torch.bfloat16)
    slots, off = [], 0
    for s, n in enumerate(lens):
        slots += [int(bt[s, t // bs]) * bs + t % bs for t in range(n)]
    cache = torch.randn(2, nb, bs, hkv, d, generator=gen).to(torch.bfloat16)
    new = oracle.kv_cache_write(k, v, torch.tensor(slots), cache)
    ks, vs = oracle.paged_gather(new, bt, torch.tensor(lens))
    for s, n in enumerate(lens):
        assert np.array_equal(ks[s], k[off:off + n].double().numpy())
        assert np.array_equal(vs[s], v[off:off + n].double().numpy())
        off += n


def test_kv_cache_write_padding_slots_and_errors():
    cache = torch.randn(2, 3, 8, 1, 32, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    k = torch.ones(3, 1, 32, dtype=torch.bfloat16)
    new = oracle.kv_cache_write(k, k, torch.tensor([-1, 9, -1]), cache)
    changed = (new != cache).any(dim=-1).any(dim=-1)
    assert changed.sum() == 2 and changed[0, 1, 1] and changed[1, 1, 1]  # only slot 9 = block 1, offset 1
    dup = oracle.kv_cache_write(torch.stack([k[0], 2 * k[0]]), torch.stack([k[0], 2 * k[0]]), torch.tensor([4, 4]), cache)
    assert torch.equal(dup[0, 0, 4], 2 * k[0])  # tokens in order: the last one stays
    with pytest.raises(ValueError):
        oracle.kv_cache_write(k, k, torch.tensor([0, 24, 1]), cache)  # 3 blocks of 8 = slots 0..23


# -------------------------------------------------------- paged prefill (f2)

def _paged_ctx(seed, lens, hq, hkv, d, bs=16):
    """A paged cache holding each sequence's contiguous K/V at a random block permutation."""
    gen = torch.Generator().manual_seed(seed)
    nb = sum(-(-n // bs) for n in lens) + 2
    perm = torch.randperm(nb, generator=gen)
    mb = max(-(-n // bs) for n in lens)
    bt = torch.full((len(lens), mb), -1, dtype=torch.int32)
    at = 0
    for s, n in enumerate(lens):
        m = -(-n // bs)
        bt[s, :m] = perm[at:at + m]
        at += m
    ks = [torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16) for n in lens]
    vs = [torch.randn(n, hkv, d, generator=gen).to(torch.bfloat16) for n in lens]
    cache = torch.full((2, nb, bs, hkv, d), float("nan"), dtype=torch.bfloat16)  # unused slots poisoned
    slots = [int(bt[s, t // bs]) * bs + t % bs for s, n in enumerate(lens) for t in range(n)]
    cache = oracle.kv_cache_write(torch.cat(ks), torch.cat(vs), torch.tensor(slots), cache)
    return ks, vs, cache, bt, torch.tensor(lens, dtype=torch.int32)


def test_paged_prefill_single_query_equals_decode():
    """q_len = 1 with the bottom-right causal rule sees the whole context: the decode."""
    lens = [1, 17, 40]
    ks, vs, cache, bt, sl = _paged_ctx(1, lens, 4, 2, 32)
    q = torch.randn(3, 4, 32, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    cu = torch.tensor([0, 1, 2, 3])
    o1, l1 = oracle.attention_paged_prefill(q, cache, bt, sl, cu, 0.2, True)
    o2, l2 = oracle.attention_paged(q, cache, bt, sl, 0.2)
    assert np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1.T, l2, rtol=0, atol=1e-12)


def test_paged_prefill_whole_context_equals_varlen_causal():
    lens = [5, 33, 16]
    ks, vs, cache, bt, sl = _paged_ctx(3, lens, 4, 1, 32)
    q = torch.randn(sum(lens), 4, 32, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    cu = workloads.cu_from_lengths(lens)
    o1, l1 = oracle.attention_paged_prefill(q, cache, bt, sl, cu, 0.3, True)
    o2, l2 = oracle.attention_varlen(q, torch.cat(ks), torch.cat(vs), cu, cu, 0.3, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_prefill_second_chunk_equals_tail_of_full_causal():
    """Chunked prefill: the last L - c queries over a context of L tokens give the
    last L - c rows of causal attention over the whole sequence."""
    L, c = 45, 19
    ks, vs, cache, bt, sl = _paged_ctx(5, [L], 2, 2, 32)
    qf = torch.randn(L, 2, 32, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    o1, l1 = oracle.attention_paged_prefill(qf[c:], cache, bt, sl, torch.tensor([0, L - c]), 0.25, True)
    o2, l2 = oracle.attention_single(qf, ks[0], vs[0], 0.25, True)
    assert np.allclose(o1, o2[c:], rtol=0, atol=1e-12) and np.allclose(l1, l2[:, c:], rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.attention_paged_prefill(qf[c:], cache, bt, sl, torch.tensor([0, L]), 0.25, True)  # cu past Tq


# ------------------------------------------------ padding mask -> varlen (f3)

def _masked_case(seed, b, s, hq, hkv, d):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(b, s, hq, d, generator=gen).to(torch.bfloat16)
    k = torch.randn(b, s, hkv, d, generator=gen).to(torch.bfloat16)
    v = torch.randn(b, s, hkv, d, generator=gen).to(torch.bfloat16)
    return q, k, v


def test_masked_prefix_mask_equals_dense_on_the_valid_prefix():
    """A mask that keeps a prefix of each row is attention over that prefix,
    zeros and -inf at the padding."""
    q, k, v = _masked_case(1, 2, 20, 2, 1, 32)
    n = [13, 20]
    mask = torch.zeros(2, 20, dtype=torch.uint8)
    for i, L in enumerate(n):
        mask[i, :L] = 1
    for causal in (False, True):
        o, l = oracle.attention_masked(q, k, v, mask, 0.3, causal)
        for i, L in enumerate(n):
            r_o, r_l = oracle.attention_single(q[i, :L], k[i, :L], v[i, :L], 0.3, causal)
            assert np.array_equal(o[i, :L], r_o) and np.array_equal(l[i][:, :L], r_l)
            assert np.all(o[i, L:] == 0) and np.all(l[i][:, L:] == -np.inf)


def test_masked_scattered_mask_is_the_packed_varlen_of_the_kept_tokens():
    q, k, v = _masked_case(2, 2, 24, 4, 2, 32)
    g = torch.Generator().manual_seed(3)
    mask = (torch.rand(2, 24, generator=g) < 0.6).to(torch.uint8)
    keep = [torch.nonzero(mask[i]).flatten() for i in range(2)]
    lens = [len(x) for x in keep]
    qp = torch.cat([q[i, keep[i]] for i in range(2)])
    kp = torch.cat([k[i, keep[i]] for i in range(2)])
    vp = torch.cat([v[i, keep[i]] for i in range(2)])
    cu = workloads.cu_from_lengths(lens)
    rv, rl = oracle.attention_varlen(qp, kp, vp, cu, cu, 0.2, True)
    o, l = oracle.attention_masked(q, k, v, mask, 0.2, True)
    for i in range(2):
        a = int(cu[i])
        assert np.array_equal(o[i, keep[i].numpy()], rv[a:a + lens[i]])
        assert np.array_equal(l[i][:, keep[i].numpy()], rl[:, a:a + lens[i]])
    assert np.all(o[mask.numpy() == 0] == 0)


def test_masked_cross_keeps_every_query():
    """Cross-attention: masked-out keys get no weight, every query row is computed."""
    q, k, v = _masked_case(4, 1, 16, 2, 2, 32)
    mask = torch.zeros(1, 16, dtype=torch.uint8)
    mask[0, [1, 4, 5, 11]] = 1
    o, l = oracle.attention_masked(q, k, v, mask, 0.25, False, cross=True)
    idx = [1, 4, 5, 11]
    r_o, r_l = oracle.attention_single(q[0], k[0, idx], v[0, idx], 0.25, False)
    assert np.array_equal(o[0], r_o) and np.array_equal(l[0], r_l)


# --------------------------------------------- block-sparse video attention (f4)

def _vsa_layout_cases():
    with open(os.path.join(GOLDEN, "vsa_layout_examples.json")) as f:
        return json.load(f)["cases"]


def _runs_to_tokens(runs):
    return [i for a, b in runs for i in range(a, b)]


@pytest.mark.parametrize("case", _vsa_layout_cases(), ids=lambda c: c["name"])
def test_vsa_blocks_match_the_hand_worked_layouts(case):
    """Block layouts worked by hand from the page's tiling functions: the
    chunking of each prefix segment on its own, the T, H, W order of the
    tiles, row-major order inside a tile, remainder tiles at the far edges."""
    blocks, n_prefix = oracle.vsa_blocks(case["prefix"], tuple(case["video"]))
    assert n_prefix == case["n_prefix_blocks"]
    assert [len(b) for b in blocks] == case["block_sizes"]
    assert [b.tolist() for b in blocks] == [_runs_to_tokens(r) for r in case["blocks"]]


def test_vsa_block_map_hand_worked_with_a_tie():
    """Prefix of 2 tokens (one block) and a 1 x 1 x 16 grid (four video blocks
    of 4 tokens).  Every query row is (1, 0); the key rows of block b are all
    (s_b, 0) with s = (5, 1, 3, 3, 2), so the block means are exact and the
    block scores at scale 1 are exactly s.  Top-1 among the video blocks is a
    tie between blocks 2 and 3, which goes to block 2 (the lower index); top-2
    takes both; the prefix key block is always kept and the prefix query block
    keeps every block."""
    blocks, n_prefix = oracle.vsa_blocks([2], (1, 1, 16))
    assert n_prefix == 1 and [len(b) for b in blocks] == [2, 4, 4, 4, 4]
    s = [5.0, 1.0, 3.0, 3.0, 2.0]
    q = torch.zeros(18, 1, 2)
    q[:, 0, 0] = 1.0
    k = torch.zeros(18, 1, 2)
    for b, rows in enumerate(blocks):
        k[torch.from_numpy(rows), 0, 0] = s[b]
    expect = {1: [True, False, True, False, False], 2: [True, False, True, True, False],
              3: [True, False, True, True, True]}
    for topk, row in expect.items():
        bm = oracle.vsa_block_map(q, k, blocks, n_prefix, topk, 1.0)[0]
        assert bm[0].all()  # the prefix query block keeps every block
        for i in range(1, 5):
            assert bm[i].tolist() == row, (topk, i)


def test_vsa_block_sparse_zero_query_is_the_mean_of_the_kept_tokens():
    """q = 0 makes every score 0, so each query token's output is the plain
    mean of V over the tokens of the key blocks its block keeps and its lse
    is ln(their count): a closed form for any block map (here one chosen by
    hand, unrelated to the scores), with GQA (head h reads KV head h // 2)."""
    blocks, n_prefix = oracle.vsa_blocks([5], (2, 3, 6))  # sizes 5, 24, 12
    assert [len(b) for b in blocks] == [5, 24, 12]
    g = torch.Generator().manual_seed(7)
    S = 41
    q = torch.zeros(S, 4, 3)
    k = torch.randn(S, 2, 3, generator=g)
    v = torch.randn(S, 2, 3, generator=g).double()
    bm = np.zeros((4, 3, 3), dtype=bool)
    bm[0] = [[1, 0, 0], [1, 1, 0], [0, 0, 1]]
    bm[1] = [[1, 1, 1], [0, 1, 0], [1, 0, 1]]
    bm[2] = [[0, 1, 1], [0, 0, 1], [1, 1, 0]]
    bm[3] = [[1, 0, 1], [1, 1, 1], [0, 1, 0]]
    out, lse = oracle.attention_block_sparse(q, k, v, blocks, bm, 0.5)
    for h in range(4):
        for i, rows in enumerate(blocks):
            keys = np.concatenate([blocks[j] for j in range(3) if bm[h, i, j]])
            mean = v[torch.from_numpy(keys), h // 2].numpy().mean(axis=0)
            assert np.allclose(out[rows, h], mean, rtol=0, atol=1e-12)
            assert np.allclose(lse[h, rows], math.log(len(keys)), rtol=0, atol=1e-12)


def test_vsa_blocks_partition_the_sequence_into_boxes():
    prefix, shape = [70, 5], (5, 6, 7)
    blocks, n_prefix = oracle.vsa_blocks(prefix, shape)
    allidx = np.concatenate(blocks)
    assert np.array_equal(np.sort(allidx), np.arange(75 + 5 * 6 * 7))  # every token exactly once
    assert [len(b) for b in blocks[:n_prefix]] == [64, 6, 5]
    # video block sizes: per-axis sizes 4,...,4,remainder multiplied out in T, H, W order
    per_axis = [[min(4, n - i) for i in range(0, n, 4)] for n in shape]
    expect = [a * b * c for a in per_axis[0] for b in per_axis[1] for c in per_axis[2]]
    assert [len(b) for b in blocks[n_prefix:]] == expect
    for b in blocks[n_prefix:]:  # each block is an axis-aligned box of the grid
        t, h, w = np.unravel_index(b - 75, shape)
        for axis in (t, h, w):
            lo, hi = axis.min(), axis.max()
            assert lo % 4 == 0 and hi - lo < 4 and set(axis) == set(range(lo, hi + 1))
        assert len(b) == len(set(t)) * len(set(h)) * len(set(w))


def _vsa_inputs(seed, prefix, shape, hq, hkv, d):
    n = sum(prefix) + int(np.prod(shape))
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, hq, d, generator=g).to(torch.bfloat16), torch.randn(n, hkv, d, generator=g).to(torch.bfloat16),
            torch.randn(n, hkv, d, generator=g).to(torch.bfloat16))


def test_vsa_keeping_every_block_is_dense_attention():
    q, k, v = _vsa_inputs(1, [20], (4, 5, 6), 4, 2, 32)
    blocks, npre = oracle.vsa_blocks([20], (4, 5, 6))
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk=100, scale=0.2)
    assert bm.all()
    o, l = oracle.attention_block_sparse(q, k, v, blocks, bm, 0.2)
    r_o, r_l = oracle.attention_single(q, k, v, 0.2, False)
    assert np.allclose(o, r_o, rtol=0, atol=1e-12) and np.allclose(l, r_l, rtol=0, atol=1e-12)


def test_vsa_top1_follows_planted_routing_and_attends_only_there():
    """Query block i's mean points at key block pi(i): top-1 keeps pi(i) (plus
    the prefix), and its rows equal attention over those keys alone."""
    prefix, shape, d = [10], (4, 8, 8), 32
    blocks, npre = oracle.vsa_blocks(prefix, shape)
    nb, nv = len(blocks), len(blocks) - npre
    n = sum(prefix) + int(np.prod(shape))
    rng = np.random.default_rng(3)
    pi = rng.permutation(nv) + npre
    q = torch.zeros(n, 1, d)
    k = torch.zeros(n, 1, d)
    for i in range(npre, nb):
        q[blocks[i], 0, pi[i - npre] % d] = 1.0
        k[blocks[i], 0, i % d] = 1.0
    q = (q + 0.01 * torch.randn(n, 1, d, generator=torch.Generator().manual_seed(4))).to(torch.bfloat16)
    k, v = k.to(torch.bfloat16), torch.randn(n, 1, d, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk=1, scale=1.0)
    for i in range(npre, nb):
        assert set(np.nonzero(bm[0, i])[0]) == set(range(npre)) | {int(pi[i - npre])}
    assert bm[0, :npre].all()  # prefix queries stay dense
    o, l = oracle.attention_block_sparse(q, k, v, blocks, bm, 1.0)
    for i in (npre, nb - 1):
        keys = np.concatenate([blocks[j] for j in range(npre)] + [blocks[pi[i - npre]]])
        r_o, r_l = oracle.attention_single(q[blocks[i]], k[keys], v[keys], 1.0, False)
        assert np.allclose(o[blocks[i]], r_o, rtol=0, atol=1e-12)
        assert np.allclose(l[:, blocks[i]], r_l, rtol=0, atol=1e-12)
    r_o, _ = oracle.attention_single(q[blocks[0]], k, v, 1.0, False)
    assert np.allclose(o[blocks[0]], r_o, rtol=0, atol=1e-12)


def test_vsa_pooling_divides_by_the_true_block_size():
    """A small edge block whose keys match best must win top-1: pooling that
    divided by 64 instead of the block's size would shrink its mean."""
    blocks, npre = oracle.vsa_blocks([], (4, 4, 6))  # blocks of 64 and 32 tokens
    assert [len(b) for b in blocks] == [64, 32]
    n, d = 96, 32
    q = torch.zeros(n, 1, d)
    q[:, 0, 0] = 1.0
    k = torch.zeros(n, 1, d)
    k[blocks[0], 0, 0] = 0.9
    k[blocks[1], 0, 0] = 1.0
    bm = oracle.vsa_block_map(q.to(torch.bfloat16), k.to(torch.bfloat16), blocks, npre, topk=1, scale=1.0)
    assert bm[0, :, 1].all() and not bm[0, :, 0].any()


def test_vsa_pool_of_a_linear_ramp_is_the_box_centre():
    """x = a + b t + c h + d w over the video grid: the mean of an axis-aligned
    box is the value at the box's centre, whatever its (edge-clipped) size;
    a prefix chunk's mean is the mean of its token positions."""
    prefix, shape = [70], (5, 6, 7)
    blocks, npre = oracle.vsa_blocks(prefix, shape)
    n = 70 + 5 * 6 * 7
    x = np.zeros((n, 2, 1))
    x[:70, 0, 0] = np.arange(70)
    t, h, w = np.meshgrid(*[np.arange(a) for a in shape], indexing="ij")
    x[70:, 0, 0] = (1.0 + 2.0 * t + 3.0 * h + 5.0 * w).ravel()
    x[:, 1, 0] = 7.0  # a constant head pools to the constant
    pooled = oracle.vsa_pool(x, blocks)
    assert pooled.shape == (len(blocks), 2, 1)
    assert np.allclose(pooled[:, 1, 0], 7.0, rtol=0, atol=0)
    assert pooled[0, 0, 0] == 31.5 and pooled[1, 0, 0] == 66.5  # chunks [0, 64) and [64, 70)
    for b in range(npre, len(blocks)):
        tt, hh, ww = np.unravel_index(blocks[b] - 70, shape)
        centre = 1.0 + 2.0 * (tt.min() + tt.max()) / 2 + 3.0 * (hh.min() + hh.max()) / 2 + 5.0 * (ww.min() + ww.max()) / 2
        assert abs(pooled[b, 0, 0] - centre) < 1e-12
