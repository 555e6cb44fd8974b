"""GPU parity: every entry point of libgbattn.so against the float64 oracle on
the same seeded bf16 inputs (max |out err| <= 1e-2 with fp32 out, max |lse
err| <= 1e-3), plus the bit-exact invariants and the device status bits."""

import math

import numpy as np
import pytest
import torch

import attention_forward_09_gb300 as gb
import oracle
import workloads
from _helpers import (LSE_TOL, OUT_TOL, assert_close, bf16_half_ulp, dev, max_err, status_word, to_np,
                      vsa_lists_from_map, vsa_map_from_lists)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_09_gb300 import _build

    _build.build()
    gb.load_library()


def _gen(seed, *shape):
    return workloads.randn_bf16(torch.Generator().manual_seed(seed), *shape)


def _dense_case(B, Sq, Sk, Hq, Hkv, D, causal, seed, scale=None, out_dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    q = workloads.randn_bf16(g, B, Sq, Hq, D)
    k = workloads.randn_bf16(g, B, Sk, Hkv, D)
    v = workloads.randn_bf16(g, B, Sk, Hkv, D)
    scale = scale or 1.0 / math.sqrt(D)
    st = status_word()
    out, lse = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), scale, causal, lse=True,
                                 out_dtype=out_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return (q, k, v, scale), out, lse


def _varlen_case(lens_q, lens_k, Hq, Hkv, D, causal, seed):
    g = torch.Generator().manual_seed(seed)
    q = workloads.randn_bf16(g, sum(lens_q), Hq, D)
    k = workloads.randn_bf16(g, sum(lens_k), Hkv, D)
    v = workloads.randn_bf16(g, sum(lens_k), Hkv, D)
    cq, ck = workloads.cu_from_lengths(lens_q), workloads.cu_from_lengths(lens_k)
    scale = 1.0 / math.sqrt(D)
    st = status_word()
    out, lse = gb.attn_fwd_varlen(q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()),
                                  max(lens_q + [0]), max(lens_k + [0]), scale, causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return (q, k, v, cq, ck, scale), out, lse


# ------------------------------------------------------------------ dense

@pytest.mark.parametrize("D", workloads.HEAD_SIZES)
@pytest.mark.parametrize("causal", [False, True])
def test_dense_all_head_sizes(D, causal):
    (q, k, v, s), out, lse = _dense_case(2, 200, 200, 4, 2, D, causal, seed=D + causal)
    ro, rl = oracle.attention_dense(q, k, v, s, causal)
    assert_close(out, lse, ro, rl, what=f"dense D={D} causal={causal}")


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (1, 300), (37, 1), (100, 300), (300, 100), (129, 127), (256, 512)])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_ragged_and_bottom_right_causal(Sq, Sk, causal):
    (q, k, v, s), out, lse = _dense_case(1, Sq, Sk, 3, 1, 128, causal, seed=Sq * 7 + Sk)
    ro, rl = oracle.attention_dense(q, k, v, s, causal)
    assert_close(out, lse, ro, rl, what=f"dense Sq={Sq} Sk={Sk} causal={causal}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (8, 1), (32, 8)])
def test_dense_gqa_ratios(Hq, Hkv):
    (q, k, v, s), out, lse = _dense_case(1, 130, 190, Hq, Hkv, 64, False, seed=Hq + 100 * Hkv)
    ro, rl = oracle.attention_dense(q, k, v, s, False)
    assert_close(out, lse, ro, rl, what=f"GQA {Hq}/{Hkv}")


def test_dense_bf16_output_within_rounding():
    (q, k, v, s), out, lse = _dense_case(1, 150, 150, 2, 2, 128, True, seed=3, out_dtype=torch.bfloat16)
    ro, rl = oracle.attention_dense(q, k, v, s, True)
    err = np.abs(to_np(out) - ro)
    assert np.all(err <= OUT_TOL + bf16_half_ulp(ro))
    assert max_err(to_np(lse), rl) <= LSE_TOL


def test_empty_keys_give_zero_and_minus_inf():
    (q, k, v, s), out, lse = _dense_case(2, 5, 0, 2, 2, 64, False, seed=1)
    assert torch.all(out == 0) and torch.all(lse == -math.inf)


def test_large_logits_rescale_path():
    """Scores spanning hundreds of log2 units force the O rescale."""
    (q, k, v, s), out, lse = _dense_case(1, 128, 512, 2, 2, 128, False, seed=9, scale=2.0)
    ro, rl = oracle.attention_dense(q, k, v, 2.0, False)
    assert_close(out, lse, ro, rl, lse_tol=5e-3, what="large logits")  # |lse| ~ 100 here


# Query tiles wholly inside their document leave through shared memory and
# TMA tiled stores; at D = 96 a bf16 row is one and a half 128-byte boxes,
# so the second box is half outside the tensor and clipped.  Causal (two-tile
# kernel): tile A, with fewer KV tiles than tile B, stores directly.

@pytest.mark.parametrize("D", [64, 96, 128, 192, 256])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("causal", [False, True])
def test_dense_tma_store_epilogue(D, out_dtype, causal):
    g = torch.Generator().manual_seed(D + 7 * causal)
    q, k, v = (workloads.randn_bf16(g, 2, n, 2, D) for n in (512, 300, 300))
    s = 1.0 / math.sqrt(D)
    out = torch.full((2, 512, 2, D), float("nan"), dtype=out_dtype, device=dev())  # unwritten stays NaN
    st = status_word()
    out, lse = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), s, causal, out=out, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle.attention_dense(q, k, v, s, causal)
    if out_dtype == torch.float32:
        assert_close(out, lse, ro, rl, what=f"TMA-store epilogue D={D} causal={causal}")
    else:
        err = np.abs(to_np(out) - ro)
        assert np.all(err <= OUT_TOL + bf16_half_ulp(ro))
        assert max_err(to_np(lse), rl) <= LSE_TOL
    assert torch.isfinite(out.float()).all()


# Dense non-causal launches of more than one wave (D <= 128) run one CTA per
# SM that walks its items in turn (on 152 SMs: 320 items = 2 or 3 per CTA),
# loading the next item's Q and K_0 during the current epilogue.

@pytest.mark.parametrize("D,out_dtype", [(128, torch.float32), (96, torch.bfloat16), (96, torch.float32),
                                         (64, torch.float32), (64, torch.bfloat16)])
def test_dense_persistent_items(D, out_dtype):
    (q, k, v, s), out, lse = _dense_case(1, 512, 300, 160, 8, D, False, seed=D + 91, out_dtype=out_dtype)
    ro, rl = oracle.attention_dense(q, k, v, s, False)
    if out_dtype == torch.float32:
        assert_close(out, lse, ro, rl, what=f"persistent D={D}")
    else:
        err = np.abs(to_np(out) - ro)
        assert np.all(err <= OUT_TOL + bf16_half_ulp(ro))
        assert max_err(to_np(lse), rl) <= LSE_TOL


def test_dense_persistent_then_split_tail():
    """328 items, 9 KV tiles: 304 on a persistent grid, then 24 split 2-way."""
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert gb.attn_fwd_dense_plan(1, 512, 1100, 164, 4, 128, False) == (2, 2)
    (q, k, v, s), out, lse = _dense_case(1, 512, 1100, 164, 4, 128, False, seed=92)
    ro, rl = oracle.attention_dense(q, k, v, s, False)
    assert_close(out, lse, ro, rl, what="persistent + split tail")


# Dense non-causal launches whose last wave would be under half full give
# those items to clusters of 2, 4 or 8 CTAs, each taking a share of the keys,
# which merge their partial softmaxes on chip.  On a 152-SM GB300 the eight
# items below split 2-, 4- and 8-way by key length (8, 17 and 33 KV tiles).

@pytest.mark.parametrize("D", [64, 96, 128])
@pytest.mark.parametrize("Sk", [1024, 2100, 4200])
def test_dense_split_tail_items(D, Sk):
    launches, split = gb.attn_fwd_dense_plan(1, 300, Sk, 4, 2, D, False)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert (launches, split) == (1, {1024: 2, 2100: 4, 4200: 8}[Sk])
    (q, k, v, s), out, lse = _dense_case(1, 300, Sk, 4, 2, D, False, seed=D * 3 + Sk)
    ro, rl = oracle.attention_dense(q, k, v, s, False)
    assert_close(out, lse, ro, rl, what=f"split tail D={D} Sk={Sk}")


def test_dense_split_after_full_waves():
    """160 items: one full wave of 152, then 8 items split 2-way."""
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert gb.attn_fwd_dense_plan(1, 256, 1100, 160, 8, 64, False) == (2, 2)
    (q, k, v, s), out, lse = _dense_case(1, 256, 1100, 160, 8, 64, False, seed=77)
    ro, rl = oracle.attention_dense(q, k, v, s, False)
    assert_close(out, lse, ro, rl, what="full wave + split tail")


def test_dense_split_bf16_output():
    (q, k, v, s), out, lse = _dense_case(2, 256, 2048, 4, 4, 128, False, seed=78, out_dtype=torch.bfloat16)
    ro, rl = oracle.attention_dense(q, k, v, s, False)
    err = np.abs(to_np(out) - ro)
    assert np.all(err <= OUT_TOL + bf16_half_ulp(ro))
    assert max_err(to_np(lse), rl) <= LSE_TOL


# ------------------------------------------------------------------ varlen

def test_tiny_varlen_config():
    w = workloads.tiny_varlen()
    (q, k, v, cq, ck, s), out, lse = _varlen_case(w.lens_q, w.lens_k, w.Hq, w.Hkv, w.D, w.causal, w.seed)
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, s, False)
    assert_close(out, lse, ro, rl, what="tiny varlen")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_odd_lengths_and_empty_docs(causal):
    lens_q = [1, 37, 0, 127, 129, 300]
    lens_k = [1, 37, 5, 127, 200, 301]
    (q, k, v, cq, ck, s), out, lse = _varlen_case(lens_q, lens_k, 8, 2, 128, causal, seed=11 + causal)
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, s, causal)
    assert_close(out, lse, ro, rl, what=f"varlen causal={causal}")


# Packed documents at every head size: both prefill kernels (two query
# tiles per CTA for D <= 128, one for D = 192 / 256) in their varlen mode,
# documents with Lq != Lk, an empty document, and lengths on both sides of
# the 128-row tile and the 256-row item.

VARLEN_EDGE_Q = [127, 128, 0, 129, 255, 257, 1, 300]
VARLEN_EDGE_K = [128, 127, 5, 129, 300, 255, 1, 257]


@pytest.mark.parametrize("D", workloads.HEAD_SIZES)
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_all_head_sizes_at_tile_boundaries(D, causal):
    (q, k, v, cq, ck, s), out, lse = _varlen_case(VARLEN_EDGE_Q, VARLEN_EDGE_K, 6, 2, D, causal, seed=3 * D + causal)
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, s, causal)
    assert_close(out, lse, ro, rl, what=f"varlen D={D} causal={causal}")


@pytest.mark.parametrize("D", [96, 192, 256])
def test_varlen_bf16_output(D):
    g = torch.Generator().manual_seed(D)
    lq, lk = [300, 128, 77], [129, 256, 300]
    q, k, v = workloads.randn_bf16(g, sum(lq), 4, D), workloads.randn_bf16(g, sum(lk), 4, D), \
        workloads.randn_bf16(g, sum(lk), 4, D)
    cq, ck = workloads.cu_from_lengths(lq), workloads.cu_from_lengths(lk)
    s = 1.0 / math.sqrt(D)
    st = status_word()
    out, lse = gb.attn_fwd_varlen(q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()), max(lq),
                                  max(lk), s, True, lse=True, out_dtype=torch.bfloat16, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, s, True)
    assert np.all(np.abs(to_np(out) - ro) <= OUT_TOL + bf16_half_ulp(ro))
    assert max_err(to_np(lse), rl) <= LSE_TOL


# No cross-document attention, whatever the neighbours hold: a document's
# last KV tile reaches into the next document's rows (or past the last
# document), and those rows are NaN or Inf here.  Every other document must
# still match the oracle.

@pytest.mark.parametrize("D", workloads.HEAD_SIZES)
@pytest.mark.parametrize("poison", [float("nan"), float("inf")])
def test_varlen_poisoned_neighbours_do_not_leak(D, poison):
    lq, lk = [100, 77, 129, 60], [130, 50, 200, 33]
    g = torch.Generator().manual_seed(D + 1)
    extra = 40  # rows of k / v (and q) past the last document
    q = workloads.randn_bf16(g, sum(lq) + extra, 4, D)
    k = workloads.randn_bf16(g, sum(lk) + extra, 2, D)
    v = workloads.randn_bf16(g, sum(lk) + extra, 2, D)
    cq, ck = workloads.cu_from_lengths(lq), workloads.cu_from_lengths(lk)
    for t, cu in ((q, cq), (k, ck), (v, ck)):
        t[int(cu[1]):int(cu[2])] = poison  # document 1
        t[int(cu[-1]):] = poison           # rows past the last document
    s = 1.0 / math.sqrt(D)
    for causal in (False, True):
        st = status_word()
        out, lse = gb.attn_fwd_varlen(q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()), max(lq),
                                      max(lk), s, causal, lse=True, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for n in (0, 2, 3):
            a, b, c, d = int(cq[n]), int(cq[n + 1]), int(ck[n]), int(ck[n + 1])
            ro, rl = oracle.attention_single(q[a:b], k[c:d], v[c:d], s, causal)
            assert_close(out[a:b], lse[:, a:b], ro, rl, what=f"document {n} D={D} causal={causal}")


@pytest.mark.parametrize("D,B,Sq,Sk,Hq,Hkv", [
    (64, 3, 200, 200, 4, 2), (96, 3, 200, 200, 4, 2), (128, 3, 200, 200, 4, 2), (192, 3, 200, 200, 4, 2),
    (256, 3, 200, 200, 4, 2),
    (128, 2, 256, 1100, 4, 2),   # the last wave split along the keys over 2-CTA clusters
    (64, 2, 256, 200, 160, 8),   # a persistent grid of one CTA per SM
])
def test_dense_poisoned_batch_entry_does_not_leak(D, B, Sq, Sk, Hq, Hkv):
    g = torch.Generator().manual_seed(D + B + Sk)
    q = workloads.randn_bf16(g, B, Sq, Hq, D)
    k = workloads.randn_bf16(g, B, Sk, Hkv, D)
    v = workloads.randn_bf16(g, B, Sk, Hkv, D)
    for t in (q, k, v):
        t[1] = float("nan")
    s = 1.0 / math.sqrt(D)
    st = status_word()
    out, lse = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), s, False, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in range(B):
        if b == 1:
            continue
        ro, rl = oracle.attention_single(q[b], k[b], v[b], s, False)
        assert_close(out[b], lse[b], ro, rl, what=f"batch {b} D={D}")


# Packed documents whose one-CTA-per-item grid would exceed a wave run on a
# persistent grid that walks the items tile-major (the heavy causal tiles of
# every document first).  The lengths include an empty document, a document
# with no keys (items with nothing to load), Lq > Lk and Lq < Lk documents.

WALK_Q = [300, 1000, 77, 2000, 0, 513, 100, 129, 257]
WALK_K = [300, 1000, 77, 2000, 9, 513, 0, 260, 128]


@pytest.mark.parametrize("D", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_persistent_walk(D, causal):
    (q, k, v, cq, ck, s), out, lse = _varlen_case(WALK_Q, WALK_K, 32, 8, D, causal, seed=5 * D + causal)
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, s, causal)
    assert_close(out, lse, ro, rl, what=f"persistent varlen D={D} causal={causal}")


def test_varlen_persistent_walk_bf16_output_and_repeat():
    g = torch.Generator().manual_seed(71)
    q, k, v = (workloads.randn_bf16(g, sum(x), h, 128) for x, h in ((WALK_Q, 16), (WALK_K, 4), (WALK_K, 4)))
    cq, ck = workloads.cu_from_lengths(WALK_Q).to(dev()), workloads.cu_from_lengths(WALK_K).to(dev())
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    st = status_word()
    outs = [gb.attn_fwd_varlen(qd, kd, vd, cq, ck, max(WALK_Q), max(WALK_K), 0.09, True, lse=True,
                               out_dtype=torch.bfloat16, dev_status=st) for _ in range(3)]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle.attention_varlen(q, k, v, cq.cpu(), ck.cpu(), 0.09, True)
    assert np.all(np.abs(to_np(outs[0][0]) - ro) <= OUT_TOL + bf16_half_ulp(ro))
    assert max_err(to_np(outs[0][1]), rl) <= LSE_TOL
    for o, l in outs[1:]:  # the same bits on every launch
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_varlen_many_short_documents():
    """More documents than the persistent walk takes: the one-CTA-per-item grid."""
    rng = np.random.default_rng(8)
    lens = [int(x) for x in rng.integers(0, 40, 600)]
    (q, k, v, cq, ck, s), out, lse = _varlen_case(lens, lens, 4, 2, 64, True, seed=72)
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, s, True)
    assert_close(out, lse, ro, rl, what="600 short documents")


def test_varlen_pack_equals_documents_alone_bit_exact():
    lens = [129, 37, 300]
    (q, k, v, cq, ck, s), out, lse = _varlen_case(lens, lens, 4, 4, 64, True, seed=5)
    for n, L in enumerate(lens):
        a, b = int(cq[n]), int(cq[n + 1])
        o1, l1 = gb.attn_fwd_varlen(q[a:b].contiguous().to(dev()), k[a:b].contiguous().to(dev()),
                                    v[a:b].contiguous().to(dev()),
                                    torch.tensor([0, L], dtype=torch.int32, device=dev()),
                                    torch.tensor([0, L], dtype=torch.int32, device=dev()), L, L, s, True, lse=True)
        torch.cuda.synchronize()
        assert torch.equal(o1, out[a:b]) and torch.equal(l1, lse[:, a:b])


def test_dense_equals_varlen_with_arange_bit_exact():
    B, S, H, D = 3, 150, 4, 128
    (q, k, v, s), out, lse = _dense_case(B, S, S, H, H, D, True, seed=21)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=dev())
    ov, lv = gb.attn_fwd_varlen(q.reshape(B * S, H, D).to(dev()), k.reshape(B * S, H, D).to(dev()),
                                v.reshape(B * S, H, D).to(dev()), cu, cu, S, S, s, True, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(ov.reshape(B, S, H, D), out)
    assert torch.equal(lv.reshape(H, B, S).permute(1, 0, 2), lse)


def test_varlen_bad_cu_seqlens_sets_status():
    q = _gen(1, 64, 2, 64).to(dev())
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device=dev())  # decreasing
    st = status_word()
    out = torch.full((64, 2, 64), 7.0, device=dev())
    gb.attn_fwd_varlen(q, q, q, cu, cu, 40, 40, 0.125, False, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gb.DEV_BAD_SEQLEN
    st.zero_()
    cu2 = torch.tensor([0, 64], dtype=torch.int32, device=dev())
    gb.attn_fwd_varlen(q, q, q, cu2, cu2, 32, 32, 0.125, False, out=out, dev_status=st)  # max_seqlen too small
    torch.cuda.synchronize()
    assert int(st.item()) & gb.DEV_BAD_SEQLEN


# ------------------------------------------------------------ invariants

def test_power_of_two_prescale_bit_exact():
    """vllm-omni flash_attn.py, FlashAttentionImpl._forward_prefix_kv_slice_npu:
    inputs divided by 2 with the scale times 4, output times 2, is exact."""
    (q, k, v, s), out, lse = _dense_case(1, 200, 260, 4, 2, 128, True, seed=31)
    o2, l2 = gb.attn_fwd_dense((q / 2).to(dev()), (k / 2).to(dev()), (v / 2).to(dev()), 4 * s, True, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o2 * 2, out) and torch.equal(l2, lse)


def test_deterministic():
    (q, k, v, s), out, lse = _dense_case(1, 300, 300, 4, 4, 96, True, seed=41)
    o2, l2 = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), s, True, lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o2, out) and torch.equal(l2, lse)


@pytest.mark.parametrize("D,causal", [(192, False), (256, True), (128, True)])
def test_deterministic_one_tile_and_walk(D, causal):
    """Repeated launches give the same bits: the one-tile kernel (D = 192,
    256, P in TMEM, many KV steps) and the persistent varlen walk (D = 128)."""
    if D == 128:
        (q, k, v, cq, ck, s), out, lse = _varlen_case(WALK_Q, WALK_K, 16, 4, D, causal, seed=43)
        args = (q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()), max(WALK_Q), max(WALK_K), s,
                causal)
        runs = [gb.attn_fwd_varlen(*args, lse=True) for _ in range(4)]
    else:
        (q, k, v, s), out, lse = _dense_case(2, 700, 1500, 8, 2, D, causal, seed=42)
        runs = [gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), s, causal, lse=True) for _ in range(4)]
    torch.cuda.synchronize()
    for o2, l2 in runs:
        assert torch.equal(o2, out) and torch.equal(l2, lse)


def test_constant_values_give_constant_output():
    """Weights sum to one.  The P V product uses P rounded to bf16 while the
    normaliser sums the fp32 weights, so this holds to 2^-8 relative, not
    exactly."""
    q, k = _gen(1, 1, 260, 4, 128), _gen(2, 1, 260, 4, 128)
    v = torch.ones(1, 260, 4, 128, dtype=torch.bfloat16)
    out, _ = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), 0.09, True)
    torch.cuda.synchronize()
    assert float((out - 1).abs().max()) <= 2.0 ** -8


def test_causal_last_row_equals_full_single_query():
    (q, k, v, s), out, lse = _dense_case(1, 77, 333, 2, 2, 128, True, seed=51)
    o1, l1 = gb.attn_fwd_dense(q[:, -1:].contiguous().to(dev()), k.to(dev()), v.to(dev()), s, False, lse=True)
    torch.cuda.synchronize()
    assert float((o1[0, 0] - out[0, -1]).abs().max()) <= 1e-5
    assert float((l1[0, :, 0] - lse[0, :, -1]).abs().max()) <= 1e-5


# ---------------------------------------------------------- full configs
# Sampled rows at the full sizes the bench times; the oracle evaluates them one by one.

def _sample_rows(n, count, seed):
    r = np.random.default_rng(seed)
    rows = set([0, n - 1, min(n - 1, 127), min(n - 1, 128)])
    rows.update(int(x) for x in r.integers(0, n, count))
    return sorted(rows)


def _check_dense_sampled(w, count=24):
    q, k, v = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), w.scale, w.causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = _sample_rows(w.Sq, count, 7)
    for b in range(w.B):
        ro, rl = oracle.attention_single(q[b], k[b], v[b], w.scale, w.causal, rows=rows)
        assert_close(out[b, rows], lse[b][:, rows], ro, rl, what=f"{w.name} batch {b}")


def test_config_dit_self_attention_sampled():
    _check_dense_sampled(workloads.dit_self())


def test_config_cross_attention_sampled():
    _check_dense_sampled(workloads.cross_attn())


@pytest.mark.parametrize("D", [64, 96, 192, 256])
def test_config_head_sweep_sampled(D):
    _check_dense_sampled(workloads.head_sweep(D), count=12)


def test_config_varlen_causal_gqa_sampled():
    w = workloads.varlen_causal_gqa()
    q, k, v, cq, ck = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_varlen(q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()),
                                  max(w.lens_q), max(w.lens_k), w.scale, True, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for n, L in enumerate(w.lens_q):
        a = int(cq[n])
        rows = _sample_rows(L, 6, n)
        ro, rl = oracle.attention_single(q[a:a + L], k[a:a + L], v[a:a + L], w.scale, True, rows=rows)
        glob = [a + r for r in rows]
        assert_close(out[glob], lse[:, glob], ro, rl, what=f"doc {n} (L={L})")


# ------------------------------------------------------------------ paged

def _paged_run(w, poison=False, bt_override=None, sl_override=None, max_len=None):
    q, cache, bt, sl = w.make()
    if bt_override is not None:
        bt = bt_override
    if sl_override is not None:
        sl = sl_override
    cache_d = cache.to(dev())
    if poison:  # slots past each sequence's end hold NaN: they must never be read into the result
        for s, n in enumerate(w.seq_lens):
            if n % 128:
                blk = int(bt[s, n // 128])
                cache_d[:, blk, n % 128:] = float("nan")
    st = status_word()
    out, lse = gb.attn_fwd_paged(q.to(dev()), cache_d, bt.to(dev()), sl.to(dev()),
                                 max_len or max(w.seq_lens), w.scale, lse=True, dev_status=st)
    torch.cuda.synchronize()
    return (q, cache, bt, sl), out, lse, int(st.item())


@pytest.mark.parametrize("D", workloads.HEAD_SIZES)
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (16, 2)])
def test_paged_small(D, Hq, Hkv):
    w = workloads.Paged("p", [1, 127, 128, 129, 700, 3000], Hq, Hkv, D, seed=D + Hq, extra_blocks=3)
    (q, cache, bt, sl), out, lse, st = _paged_run(w, poison=True)
    assert st == 0
    ro, rl = oracle.attention_paged(q, cache, bt, sl, w.scale)
    assert_close(out, lse, ro, rl, what=f"paged D={D} {Hq}/{Hkv}")


def test_paged_long_context_many_splits():
    w = workloads.Paged("p", [32768, 5000, 1], 32, 8, 128, seed=77)
    (q, cache, bt, sl), out, lse, st = _paged_run(w)
    assert st == 0
    ro, rl = oracle.attention_paged(q, cache, bt, sl, w.scale)
    assert_close(out, lse, ro, rl, what="paged long")


def test_paged_block_permutation_bit_identical():
    w = workloads.Paged("p", [900, 2000, 130], 8, 2, 128, seed=5)
    (q, cache, bt, sl), out, lse, _ = _paged_run(w)
    # move every block to a new physical place and rewrite the table to match
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(99))
    cache2 = torch.empty_like(cache)
    cache2[:, perm] = cache
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].to(torch.int32), bt)
    st = status_word()
    out2, lse2 = gb.attn_fwd_paged(q.to(dev()), cache2.to(dev()), bt2.to(dev()), sl.to(dev()), max(w.seq_lens),
                                   w.scale, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert torch.equal(out2, out) and torch.equal(lse2, lse)


def test_paged_matches_dense_single_query():
    w = workloads.Paged("p", [1000, 257], 8, 2, 128, seed=15)
    (q, cache, bt, sl), out, lse, _ = _paged_run(w)
    ks, vs = oracle.paged_gather(cache, bt, sl)
    for s, n in enumerate(w.seq_lens):
        kk = torch.from_numpy(ks[s]).to(torch.bfloat16)[None].contiguous()
        vv = torch.from_numpy(vs[s]).to(torch.bfloat16)[None].contiguous()
        o1, l1 = gb.attn_fwd_dense(q[s][None, None].contiguous().to(dev()), kk.to(dev()), vv.to(dev()), w.scale,
                                   False, lse=True)
        torch.cuda.synchronize()
        assert float((o1[0, 0] - out[s]).abs().max()) <= 2e-3
        assert float((l1[0, :, 0] - lse[s]).abs().max()) <= 1e-4


def test_paged_bad_block_and_seq_len_status():
    w = workloads.Paged("p", [300, 200], 4, 2, 64, seed=3)
    q, cache, bt, sl = w.make()
    bt_bad = bt.clone()
    bt_bad[0, 1] = w.num_blocks + 5
    (_, _, _, _), out, lse, st = _paged_run(w, bt_override=bt_bad)
    assert st & gb.DEV_BAD_INDEX
    # the bad block's tokens are skipped: sequence 0 then equals attention over its other tokens
    ks, vs = oracle.paged_gather(cache, bt, sl)
    keep = np.r_[0:128, 256:300]
    ro, rl = oracle.attention_single(q[0:1], ks[0][keep], vs[0][keep], w.scale, False)
    assert_close(out[0:1], lse[0:1].T, ro, rl, what="bad block skipped")
    sl_bad = sl.clone()
    sl_bad[1] = 5000
    (_, _, _, _), out, lse, st = _paged_run(w, sl_override=sl_bad, max_len=300)
    assert st & gb.DEV_BAD_SEQLEN


def test_paged_zero_length_sequence():
    w = workloads.Paged("p", [0, 50], 4, 4, 128, seed=8)
    (q, cache, bt, sl), out, lse, st = _paged_run(w)
    assert torch.all(out[0] == 0) and torch.all(lse[0] == -math.inf)
    ro, rl = oracle.attention_paged(q, cache, bt, sl, w.scale)
    assert_close(out, lse, ro, rl, what="zero length")


def test_config_paged_decode_sampled():
    w = workloads.paged_decode()
    (q, cache, bt, sl), out, lse, st = _paged_run(w)
    assert st == 0
    pick = sorted({0, int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens)), 17, 63})
    ro, rl = oracle.attention_paged(q[pick], cache, bt[pick], sl[pick], w.scale)
    assert_close(out[pick], lse[pick], ro, rl, what="paged decode config")


def test_paged_repeated_launches_stable():
    """The decode workload launched back to back, as the bench does: no
    pipeline wait may time out and every launch gives the same bits."""
    w = workloads.paged_decode()
    q, cache, bt, sl = w.make(chunk_rows=256)
    qd, cd, btd, sld = q.to(dev()), cache.to(dev()), bt.to(dev()), sl.to(dev())
    st = status_word()
    ws = torch.empty(gb.attn_fwd_paged_workspace_size(len(w.seq_lens), w.Hq, w.Hkv, w.D, max(w.seq_lens)),
                     dtype=torch.uint8, device=dev())
    ref = None
    for _ in range(12):
        out, lse = gb.attn_fwd_paged(qd, cd, btd, sld, max(w.seq_lens), w.scale, lse=True, workspace=ws,
                                     dev_status=st)
        if ref is None:
            torch.cuda.synchronize()
            ref = (out.clone(), lse.clone())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


def test_dense_repeated_launches_stable():
    w = workloads.dit_self()
    q, k, v = w.make()
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    st = status_word()
    ref = None
    for _ in range(12):
        out, lse = gb.attn_fwd_dense(qd, kd, vd, w.scale, False, lse=True, dev_status=st)
        if ref is None:
            torch.cuda.synchronize()
            ref = (out.clone(), lse.clone())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


# ------------------------------------------------------------- KV cache write
# attn_kv_cache_write against the oracle's kv_cache_write: a copy, so bit-exact.

def _cache_write_case(seed, T, nb, bs, hkv, d, pad_every=0):
    g = torch.Generator().manual_seed(seed)
    k = workloads.randn_bf16(g, T, hkv, d)
    v = workloads.randn_bf16(g, T, hkv, d)
    cache = workloads.randn_bf16(g, 2, nb, bs, hkv, d)
    slots = torch.randperm(nb * bs, generator=g)[:T].to(torch.int32)
    if pad_every:
        slots[::pad_every] = -1  # padding tokens
    return k, v, slots, cache


@pytest.mark.parametrize("T,nb,bs,hkv,d", [(1000, 16, 128, 8, 128), (77, 9, 16, 2, 64), (300, 4, 128, 1, 256),
                                            (129, 3, 128, 4, 96), (500, 8, 128, 2, 192)])
def test_kv_cache_write_bit_exact(T, nb, bs, hkv, d):
    k, v, slots, cache = _cache_write_case(T + d, T, nb, bs, hkv, d, pad_every=7)
    ref = oracle.kv_cache_write(k, v, slots, cache)
    cd = cache.to(dev())
    st = status_word()
    gb.attn_kv_cache_write(k.to(dev()), v.to(dev()), slots.to(dev()), cd, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(cd.cpu().view(torch.int16), ref.view(torch.int16))


def test_kv_cache_write_slot_past_cache_sets_status():
    k, v, slots, cache = _cache_write_case(3, 40, 4, 16, 2, 64)
    slots[5] = 4 * 16  # one past the last slot
    cd = cache.to(dev())
    st = status_word()
    gb.attn_kv_cache_write(k.to(dev()), v.to(dev()), slots.to(dev()), cd, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gb.DEV_BAD_INDEX
    keep = slots.clone()
    keep[5] = -1  # the oracle refuses such a slot; the kernel skips it
    assert torch.equal(cd.cpu().view(torch.int16), oracle.kv_cache_write(k, v, keep, cache).view(torch.int16))


def test_kv_cache_write_then_paged_decode():
    """New tokens written through slot_mapping = block_table[s, t // 128] * 128 + t % 128
    are what attn_fwd_paged then reads: its output equals the oracle on contiguous K/V."""
    w = workloads.Paged("write_then_decode", [300, 1, 1000, 129], 8, 2, 128, seed=31, extra_blocks=2)
    q, cache, bt, sl = w.make()
    g = torch.Generator().manual_seed(32)
    ks = [workloads.randn_bf16(g, n, w.Hkv, w.D) for n in w.seq_lens]
    vs = [workloads.randn_bf16(g, n, w.Hkv, w.D) for n in w.seq_lens]
    slots = torch.tensor([int(bt[s, t // 128]) * 128 + t % 128 for s, n in enumerate(w.seq_lens) for t in range(n)],
                         dtype=torch.int32)
    cd = torch.zeros_like(cache).to(dev())
    gb.attn_kv_cache_write(torch.cat(ks).to(dev()), torch.cat(vs).to(dev()), slots.to(dev()), cd)
    st = status_word()
    out, lse = gb.attn_fwd_paged(q.to(dev()), cd, bt.to(dev()), sl.to(dev()), max(w.seq_lens), w.scale, lse=True,
                                 dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for s in range(len(w.seq_lens)):
        ro, rl = oracle.attention_single(q[s:s + 1], ks[s], vs[s], w.scale, False)
        assert_close(out[s:s + 1], lse[s:s + 1].T, ro, rl, what=f"sequence {s}")


# ------------------------------------------- prefill over the paged cache (f2)
# Several query tokens per sequence (the last q_len of its context) read their
# keys through the block table; cache slots past each seq_len hold NaN.

def _paged_prefill_run(seed, ctx, qlens, hq, hkv, d, causal, bt_override=None):
    w = workloads.Paged(f"paged_prefill_{seed}", ctx, hq, hkv, d, seed=seed, extra_blocks=2)
    _, cache, bt, sl = w.make()
    if bt_override is not None:
        bt = bt_override(bt)
    cache_d = cache.to(dev())
    for s, n in enumerate(ctx):
        if n % 128:
            cache_d[:, int(bt[s, n // 128]), n % 128:] = float("nan")
    q = workloads.randn_bf16(torch.Generator().manual_seed(seed + 7), sum(qlens), hq, d)
    cu = workloads.cu_from_lengths(qlens)
    st = status_word()
    out, lse = gb.attn_fwd_paged_prefill(q.to(dev()), cache_d, bt.to(dev()), sl.to(dev()), cu.to(dev()), max(qlens),
                                         max(ctx), w.scale, causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    return (q, cache, bt, sl, cu, w.scale), out, lse, int(st.item())


@pytest.mark.parametrize("D,hq,hkv,causal,ctx,qlens", [
    (128, 8, 2, True, [300, 1, 1000, 129], [16, 1, 200, 129]),   # spec decode, decode, chunk, whole context
    (64, 4, 4, True, [2000, 37], [300, 5]),
    (96, 4, 2, False, [500, 700], [3, 16]),
    (192, 4, 4, True, [400, 130], [130, 7]),
    (256, 2, 1, True, [260], [260]),
    (128, 4, 4, True, [50], [80]),                                # more queries than keys: leading rows see none
    (128, 8, 1, True, [700, 3000, 129], [16, 16, 5]),             # GQA packing, 16 tokens x 8 heads per tile
    (64, 16, 2, False, [900, 260], [300, 40]),                    # GQA packing, 16 x 8, several tile pairs
])
def test_paged_prefill_matches_oracle(D, hq, hkv, causal, ctx, qlens):
    (q, cache, bt, sl, cu, s), out, lse, st = _paged_prefill_run(D + len(ctx), ctx, qlens, hq, hkv, D, causal)
    assert st == 0
    ro, rl = oracle.attention_paged_prefill(q, cache, bt, sl, cu, s, causal)
    assert_close(out, lse, ro, rl, what=f"paged prefill D={D}")


def test_paged_prefill_bad_block_sets_status():
    def corrupt(bt):
        bt = bt.clone()
        bt[0, 1] = 10 ** 6
        return bt
    _, _, _, st = _paged_prefill_run(5, [300, 200], [20, 200], 4, 4, 128, True, bt_override=corrupt)
    assert st & gb.DEV_BAD_INDEX


def test_config_chunked_prefill_sampled():
    """The bench's chunked-prefill workload at full size, sampled rows of the
    shortest and the longest sequence against the oracle."""
    w = workloads.chunked_prefill()
    q, cache, bt, sl, cu = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_paged_prefill(q.to(dev()), cache.to(dev()), bt.to(dev()), sl.to(dev()), cu.to(dev()),
                                         max(w.q_lens), max(w.seq_lens), w.scale, True, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for s in (min(range(len(w.seq_lens)), key=lambda i: w.seq_lens[i]),
              max(range(len(w.seq_lens)), key=lambda i: w.seq_lens[i])):
        a, b = int(cu[s]), int(cu[s + 1])
        ks, vs = oracle.paged_gather(cache, bt[s:s + 1], sl[s:s + 1])
        rows = _sample_rows(b - a, 6, s)
        ro, rl = oracle.attention_single(q[a:b], ks[0], vs[0], w.scale, True, rows=rows)
        glob = [a + r for r in rows]
        assert_close(out[glob], lse[:, glob], ro, rl, what=f"chunked prefill sequence {s}")


# ----------------------------------------------- padding mask -> varlen (f3)

def test_mask_to_varlen_indices_bit_exact():
    g = torch.Generator().manual_seed(8)
    mask = (torch.rand(5, 3000, generator=g) < 0.55).to(torch.uint8)
    mask[2] = 0  # a row with no token at all
    cu, pos = gb.attn_mask_to_varlen(mask.to(dev()))
    torch.cuda.synchronize()
    counts = mask.sum(dim=1)
    ref_cu = torch.zeros(6, dtype=torch.int64)
    ref_cu[1:] = torch.cumsum(counts, 0)
    flat = mask.flatten().to(torch.int64)
    ref_pos = torch.where(flat != 0, torch.cumsum(flat, 0) - 1, torch.full_like(flat, -1))
    assert torch.equal(cu.cpu().to(torch.int64), ref_cu) and torch.equal(pos.cpu().to(torch.int64), ref_pos)


def test_pack_rows_zeroes_the_tail_and_round_trips():
    g = torch.Generator().manual_seed(9)
    B, S = 3, 500
    x = workloads.randn_bf16(g, B, S, 2, 64)
    mask = (torch.rand(B, S, generator=g) < 0.4).to(torch.uint8)
    xd = x.to(dev())
    xd[mask.to(dev()) == 0] = float("nan")  # padding rows must never be copied
    cu, pos = gb.attn_mask_to_varlen(mask.to(dev()))
    packed = gb.attn_pack_rows(xd, pos, cu)
    back = gb.attn_unpack_rows(packed, pos, B, S)
    torch.cuda.synchronize()
    total = int(mask.sum())
    keep = mask.flatten() != 0
    assert torch.equal(packed[:total].cpu().view(torch.int16), x.flatten(0, 1)[keep].view(torch.int16))
    assert torch.all(packed[total:].cpu() == 0)
    ref = torch.where(mask[..., None, None] != 0, x, torch.zeros_like(x))
    assert torch.equal(back.cpu().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("kind,causal,D,hq,hkv,S", [
    ("scattered", False, 128, 4, 2, 300), ("scattered", True, 64, 4, 4, 257), ("prefix", True, 128, 2, 1, 400),
    ("empty_row", False, 96, 2, 2, 200), ("cross", False, 128, 4, 4, 77)])
def test_masked_matches_oracle(kind, causal, D, hq, hkv, S):
    g = torch.Generator().manual_seed(D + S)
    B, Sq = 3, (200 if kind == "cross" else S)
    q = workloads.randn_bf16(g, B, Sq, hq, D)
    k = workloads.randn_bf16(g, B, S, hkv, D)
    v = workloads.randn_bf16(g, B, S, hkv, D)
    if kind == "prefix":
        mask = torch.zeros(B, S, dtype=torch.uint8)
        for i, n in enumerate([S, S // 2, 13]):
            mask[i, :n] = 1
    else:
        mask = (torch.rand(B, S, generator=g) < 0.65).to(torch.uint8)
        if kind == "empty_row":
            mask[1] = 0
    st = status_word()
    out, lse = gb.attn_fwd_masked(q.to(dev()), k.to(dev()), v.to(dev()), mask.to(dev()), 1.0 / math.sqrt(D), causal,
                                  cross=(kind == "cross"), lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle.attention_masked(q, k, v, mask, 1.0 / math.sqrt(D), causal, cross=(kind == "cross"))
    assert_close(out, lse, ro, rl, what=f"masked {kind}")


# Right-padded batches through attn_fwd_padded: the same results as the
# unpad -> varlen -> pad pipeline (the oracle's attention_masked) for a mask
# that keeps each row's first tokens, with NaN in every padded row (it must
# never reach a result).

PAD_LENS = [[300, 129, 0, 1], [257, 256, 255, 128], [127, 300, 13, 200]]


def _prefix_mask(lens, S):
    mask = torch.zeros(len(lens), S, dtype=torch.uint8)
    for i, n in enumerate(lens):
        mask[i, :n] = 1
    return mask


@pytest.mark.parametrize("D", workloads.HEAD_SIZES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind", ["self", "cross"])
def test_padded_matches_the_masked_oracle(D, causal, kind):
    S = 300
    lens = PAD_LENS[(D // 32 + causal) % 3]
    B, Sq = len(lens), (200 if kind == "cross" else S)
    g = torch.Generator().manual_seed(D + 3 * causal + (kind == "cross"))
    q = workloads.randn_bf16(g, B, Sq, 4, D)
    k = workloads.randn_bf16(g, B, S, 2, D)
    v = workloads.randn_bf16(g, B, S, 2, D)
    mask = _prefix_mask(lens, S)
    ro, rl = oracle.attention_masked(q, k, v, mask, 1.0 / math.sqrt(D), causal, cross=(kind == "cross"))
    for i, n in enumerate(lens):  # padding rows hold NaN: never read into a result
        k[i, n:] = float("nan")
        v[i, n:] = float("nan")
        if kind == "self":
            q[i, n:] = float("nan")
    L = torch.tensor(lens, dtype=torch.int32, device=dev())
    st = status_word()
    out, lse = gb.attn_fwd_padded(q.to(dev()), k.to(dev()), v.to(dev()), L if kind == "self" else None, L,
                                  1.0 / math.sqrt(D), causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out, lse, ro, rl, what=f"padded {kind} D={D} causal={causal}")


@pytest.mark.parametrize("D,Sk", [(128, 1100), (64, 300)])
def test_padded_split_and_persistent_paths(D, Sk):
    """Many heads (a persistent grid) and a partly filled last wave (its
    items split along the keys over a cluster): rows padded at every place."""
    g = torch.Generator().manual_seed(D + Sk)
    B, S, H = 2, 512, 160 if D == 64 else 4
    lens_q, lens_k = [512, 300], [Sk, 700 if Sk > 700 else 150]
    q = workloads.randn_bf16(g, B, S, H, D)
    k = workloads.randn_bf16(g, B, Sk, H // 4, D)
    v = workloads.randn_bf16(g, B, Sk, H // 4, D)
    s = 1.0 / math.sqrt(D)
    st = status_word()
    out, lse = gb.attn_fwd_padded(q.to(dev()), k.to(dev()), v.to(dev()),
                                  torch.tensor(lens_q, dtype=torch.int32, device=dev()),
                                  torch.tensor(lens_k, dtype=torch.int32, device=dev()), s, False, lse=True,
                                  dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for b in range(B):
        ro, rl = oracle.attention_single(q[b, :lens_q[b]], k[b, :lens_k[b]], v[b, :lens_k[b]], s, False)
        assert_close(out[b, :lens_q[b]], lse[b][:, :lens_q[b]], ro, rl, what=f"padded batch {b}")
        assert torch.all(out[b, lens_q[b]:] == 0) and torch.all(lse[b][:, lens_q[b]:] == -math.inf)


@pytest.mark.parametrize("lens_q,lens_k", [([0, 512, 100], [512, 512, 0]), ([512, 0, 257], [200, 512, 300])])
def test_padded_persistent_runs_of_empty_items(lens_q, lens_k):
    """A persistent grid (160 heads) over batch entries that are wholly or
    partly padding: long runs of items that stage nothing between items that
    do, and items whose second tile lies in the padding."""
    g = torch.Generator().manual_seed(sum(lens_q))
    B, S, H, D = 3, 512, 160, 64
    q = workloads.randn_bf16(g, B, S, H, D)
    k = workloads.randn_bf16(g, B, S, H // 8, D)
    v = workloads.randn_bf16(g, B, S, H // 8, D)
    s = 1.0 / math.sqrt(D)
    for causal in (False, True):
        st = status_word()
        out, lse = gb.attn_fwd_padded(q.to(dev()), k.to(dev()), v.to(dev()),
                                      torch.tensor(lens_q, dtype=torch.int32, device=dev()),
                                      torch.tensor(lens_k, dtype=torch.int32, device=dev()), s, causal, lse=True,
                                      dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for b in range(B):
            ro, rl = oracle.attention_single(q[b, :lens_q[b]], k[b, :lens_k[b]], v[b, :lens_k[b]], s, causal)
            assert_close(out[b, :lens_q[b]], lse[b][:, :lens_q[b]], ro, rl, what=f"entry {b} causal={causal}")
            assert torch.all(out[b, lens_q[b]:] == 0) and torch.all(lse[b][:, lens_q[b]:] == -math.inf)


def test_padded_bad_length_sets_status():
    q = _gen(1, 2, 64, 2, 64).to(dev())
    st = status_word()
    gb.attn_fwd_padded(q, q, q, torch.tensor([64, 70], dtype=torch.int32, device=dev()), None, 0.1, False,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gb.DEV_BAD_SEQLEN


def test_masked_bf16_output():
    g = torch.Generator().manual_seed(10)
    q, k, v = (workloads.randn_bf16(g, 2, 256, 2, 128) for _ in range(3))
    mask = (torch.rand(2, 256, generator=g) < 0.5).to(torch.uint8)
    out, _ = gb.attn_fwd_masked(q.to(dev()), k.to(dev()), v.to(dev()), mask.to(dev()), 0.088, False,
                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ro, _ = oracle.attention_masked(q, k, v, mask, 0.088, False)
    assert np.all(np.abs(to_np(out) - ro) <= OUT_TOL + bf16_half_ulp(ro))


def test_config_spec_decode_sampled():
    """The bench's speculative-decode workload at full size (GQA-packed tiles):
    every row of three sequences against the oracle."""
    w = workloads.spec_decode()
    q, cache, bt, sl, cu = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_paged_prefill(q.to(dev()), cache.to(dev()), bt.to(dev()), sl.to(dev()), cu.to(dev()),
                                         max(w.q_lens), max(w.seq_lens), w.scale, True, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for s in (0, 17, len(w.seq_lens) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        ks, vs = oracle.paged_gather(cache, bt[s:s + 1], sl[s:s + 1])
        ro, rl = oracle.attention_single(q[a:b], ks[0], vs[0], w.scale, True)
        assert_close(out[a:b], lse[:, a:b], ro, rl, what=f"spec decode sequence {s}")


# ------------------------------------------------- block-sparse video attention
def _vsa_inputs(seed, prefix, video, hq, hkv, d):
    n = sum(prefix) + int(np.prod(video))
    g = torch.Generator().manual_seed(seed)
    return (workloads.randn_bf16(g, n, hq, d), workloads.randn_bf16(g, n, hkv, d),
            workloads.randn_bf16(g, n, hkv, d))


def _vsa_check_map(bm_gpu, q, k, blocks, npre, topk, scale, heads=None):
    """GPU block map against the oracle's: rows whose topk-th and (topk+1)-th
    oracle scores are more than 1e-5 apart must be equal; the others must be
    a valid choice (prefix kept, topk video blocks, none worse than a block
    left out by more than 1e-5).  Returns the oracle map of the heads."""
    heads = list(range(q.shape[1])) if heads is None else heads
    g = q.shape[1] // k.shape[1]
    nb = len(blocks)
    keep = min(topk, nb - npre)
    ref = np.zeros((len(heads), nb, nb), dtype=bool)
    for x, h in enumerate(heads):
        qh, kh = q[:, h:h + 1], k[:, h // g:h // g + 1]
        ref[x] = oracle.vsa_block_map(qh, kh, blocks, npre, topk, scale)[0]
        sc = scale * oracle.vsa_pool(qh, blocks)[:, 0, :] @ oracle.vsa_pool(kh, blocks)[:, 0, :].T
        for i in range(nb):
            if np.array_equal(bm_gpu[x, i], ref[x, i]):
                continue
            assert i >= npre and keep < nb - npre, f"head {h} dense row {i} differs"
            s = np.sort(sc[i, npre:])[::-1]
            assert s[keep - 1] - s[keep] <= 1e-5, f"head {h} row {i}: unambiguous top-{keep} differs"
            chosen = bm_gpu[x, i, npre:]
            assert bm_gpu[x, i, :npre].all() and chosen.sum() == keep
            assert sc[i, npre:][chosen].min() >= sc[i, npre:][~chosen].max() - 1e-5
    return ref


@pytest.mark.parametrize("D", [64, 128])
def test_vsa_gather_and_pool_match_the_oracle(D):
    prefix, video = [100, 37], (5, 9, 10)
    q, _, _ = _vsa_inputs(60, prefix, video, 4, 2, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    assert plan.num_blocks == len(blocks) == 21 and plan.num_prefix_blocks == npre
    st = status_word()
    qt = gb.attn_gather_rows(q.to(dev()), plan.tile_index, dev_status=st)
    pooled = gb.attn_vsa_pool(qt, plan.block_sizes, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qt_h = qt.cpu()
    for b, rows in enumerate(blocks):  # bit-exact rows, zeros at the padding
        assert torch.equal(qt_h[64 * b:64 * b + len(rows)], q[torch.from_numpy(rows)])
        assert not qt_h[64 * b + len(rows):64 * b + 64].any()
    assert not qt_h[64 * len(blocks):].any()  # the odd count's empty partner block
    ref = oracle.vsa_pool(q, blocks)  # [nb, H, D]
    assert np.max(np.abs(to_np(pooled).transpose(1, 0, 2) - ref)) <= 1e-5


@pytest.mark.parametrize("prefix,video,hq,hkv,D,topk", [
    ([100, 37], (5, 9, 10), 4, 2, 128, 5),
    ([100, 37], (5, 9, 10), 4, 2, 64, 1),
    ([], (8, 12, 12), 2, 2, 128, 7),      # no prefix, 18 full blocks, even count
    ([64], (4, 8, 8), 2, 1, 128, 100),    # topk above the video block count: every block kept
])
def test_vsa_block_map_matches_the_oracle(prefix, video, hq, hkv, D, topk):
    q, k, _ = _vsa_inputs(61, prefix, video, hq, hkv, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    scale = 1.0 / math.sqrt(D)
    st = status_word()
    pq = gb.attn_vsa_pool(gb.attn_gather_rows(q.to(dev()), plan.tile_index), plan.block_sizes)
    pk = gb.attn_vsa_pool(gb.attn_gather_rows(k.to(dev()), plan.tile_index), plan.block_sizes)
    kv_list, kv_num = gb.attn_vsa_block_map(pq, pk, plan.block_sizes, npre, topk, scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sizes = [len(b) for b in blocks]
    bm = vsa_map_from_lists(kv_list, kv_num, len(blocks), npre, topk, sizes)
    _vsa_check_map(bm, q, k, blocks, npre, topk, scale)


def test_vsa_block_map_with_fewer_query_blocks_per_cta():
    """6000 video blocks: the scores of eight query blocks against every key
    block no longer fit in shared memory, so the kernel takes four per CTA."""
    prefix, video, hq, hkv, D, topk = [], (4, 240, 400), 1, 1, 64, 8
    q, k, _ = _vsa_inputs(66, prefix, video, hq, hkv, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    assert len(blocks) == 6000
    scale = 1.0 / math.sqrt(D)
    st = status_word()
    pq = gb.attn_vsa_pool(gb.attn_gather_rows(q.to(dev()), plan.tile_index), plan.block_sizes)
    pk = gb.attn_vsa_pool(gb.attn_gather_rows(k.to(dev()), plan.tile_index), plan.block_sizes)
    kv_list, kv_num = gb.attn_vsa_block_map(pq, pk, plan.block_sizes, npre, topk, scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bm = vsa_map_from_lists(kv_list, kv_num, len(blocks), npre, topk, [len(b) for b in blocks])
    _vsa_check_map(bm, q, k, blocks, npre, topk, scale)


@pytest.mark.parametrize("prefix,video,hq,hkv,D,topk,out_dtype,tiled", [
    ([100, 37], (5, 9, 10), 4, 2, 128, 5, torch.float32, False),
    ([100, 37], (5, 9, 10), 4, 2, 128, 5, torch.bfloat16, False),
    ([100, 37], (5, 9, 10), 2, 2, 64, 3, torch.float32, False),
    ([], (8, 12, 12), 2, 1, 128, 7, torch.float32, True),
    ([64], (4, 8, 8), 2, 1, 64, 100, torch.float32, False),
])
def test_vsa_fwd_matches_the_oracle_on_the_oracle_map(prefix, video, hq, hkv, D, topk, out_dtype, tiled):
    """The attention kernel alone, fed the oracle's own block map."""
    q, k, v = _vsa_inputs(62, prefix, video, hq, hkv, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    scale = 1.0 / math.sqrt(D)
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk, scale)
    ref_o, ref_l = oracle.attention_block_sparse(q, k, v, blocks, bm, scale)
    kv_list, kv_num = (x.to(dev()) for x in vsa_lists_from_map(bm, [len(b) for b in blocks], npre, topk))
    qt, kt, vt = (gb.attn_gather_rows(x.to(dev()), plan.tile_index) for x in (q, k, v))
    st = status_word()
    S = plan.tokens
    out, lse = gb.attn_fwd_vsa(qt, kt, vt, kv_list, kv_num, plan.num_blocks, npre, topk,
                               out_index=None if tiled else plan.tile_index, out_rows=None if tiled else S,
                               softmax_scale=scale, lse=True, out_dtype=out_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if tiled:  # rows stay in the tiled layout: take each token's row back out
        idx = plan.tile_index.cpu().numpy()
        tok = np.nonzero(idx >= 0)[0]
        o = np.zeros((S, hq, D))
        o[idx[tok]] = to_np(out)[tok]
        l = np.zeros((hq, S))
        l[:, idx[tok]] = to_np(lse)[:, tok]
        out, lse = o, l
    tol = OUT_TOL if out_dtype == torch.float32 else OUT_TOL + float(np.max(bf16_half_ulp(ref_o)))
    assert_close(out, lse, ref_o, ref_l, out_tol=tol, what="vsa fwd")


@pytest.mark.parametrize("D", [64, 128])
def test_vsa_fwd_padding_rows_are_never_used(D):
    """The padding rows of every 64-row block (past its token count) and the
    odd count's empty partner block hold NaN: the result is unchanged."""
    prefix, video, hq, hkv, topk = [100, 37], (5, 9, 10), 4, 2, 5
    q, k, v = _vsa_inputs(65, prefix, video, hq, hkv, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    scale = 1.0 / math.sqrt(D)
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk, scale)
    ref_o, ref_l = oracle.attention_block_sparse(q, k, v, blocks, bm, scale)
    kv_list, kv_num = (x.to(dev()) for x in vsa_lists_from_map(bm, [len(b) for b in blocks], npre, topk))
    pad = (plan.tile_index < 0).to(dev())
    qt, kt, vt = (gb.attn_gather_rows(x.to(dev()), plan.tile_index) for x in (q, k, v))
    for t in (qt, kt, vt):
        t[pad] = float("nan")
    st = status_word()
    out, lse = gb.attn_fwd_vsa(qt, kt, vt, kv_list, kv_num, plan.num_blocks, npre, topk, out_index=plan.tile_index,
                               out_rows=plan.tokens, softmax_scale=scale, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out, lse, ref_o, ref_l, what="vsa fwd, NaN padding rows")


def test_vsa_end_to_end_matches_the_oracle():
    prefix, video, hq, hkv, D, topk = [100, 37], (5, 9, 10), 4, 2, 128, 5
    q, k, v = _vsa_inputs(63, prefix, video, hq, hkv, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    scale = 1.0 / math.sqrt(D)
    st = status_word()
    out, lse = gb.attn_vsa(q.to(dev()), k.to(dev()), v.to(dev()), plan, topk, scale, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk, scale)
    ref_o, ref_l = oracle.attention_block_sparse(q, k, v, blocks, bm, scale)
    assert_close(out, lse, ref_o, ref_l, what="vsa end to end")


def test_vsa_bad_list_entry_sets_status():
    prefix, video, D, topk = [], (4, 8, 8), 128, 1
    q, k, v = _vsa_inputs(64, prefix, video, 2, 2, D)
    plan = gb.VsaPlan(prefix, video, dev())
    blocks, npre = oracle.vsa_blocks(prefix, video)
    bm = oracle.vsa_block_map(q, k, blocks, npre, topk, 0.1)
    kv_list, kv_num = (x.to(dev()) for x in vsa_lists_from_map(bm, [len(b) for b in blocks], npre, topk))
    kv_list[0] = (len(blocks) + 5) << 9 | 64 << 2 | 1  # a block past the end
    qt, kt, vt = (gb.attn_gather_rows(x.to(dev()), plan.tile_index) for x in (q, k, v))
    st = status_word()
    gb.attn_fwd_vsa(qt, kt, vt, kv_list, kv_num, plan.num_blocks, npre, topk, out_index=plan.tile_index,
                    out_rows=plan.tokens, softmax_scale=0.1, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & gb.DEV_BAD_INDEX


def test_config_vsa_video_sampled():
    """The full-size video workload: the whole device path, its block map
    checked on two heads, and rows of sampled query blocks against the oracle."""
    w = workloads.vsa_video()
    q, k, v = w.make()
    plan = gb.VsaPlan(w.prefix, w.video, dev())
    blocks, npre = oracle.vsa_blocks(w.prefix, w.video)
    st = status_word()
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    qt, kt, vt = (gb.attn_gather_rows(x, plan.tile_index, dev_status=st) for x in (qd, kd, vd))
    pq, pk = gb.attn_vsa_pool(qt, plan.block_sizes, st), gb.attn_vsa_pool(kt, plan.block_sizes, st)
    kv_list, kv_num = gb.attn_vsa_block_map(pq, pk, plan.block_sizes, npre, w.topk, w.scale, dev_status=st)
    out, lse = gb.attn_fwd_vsa(qt, kt, vt, kv_list, kv_num, plan.num_blocks, npre, w.topk,
                               out_index=plan.tile_index, out_rows=w.tokens, softmax_scale=w.scale, lse=True,
                               dev_status=st)
    out2, lse2 = gb.attn_vsa(qd, kd, vd, plan, w.topk, w.scale, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)  # the composed call is the same launches
    heads = [0, w.Hq - 1]
    sizes = [len(b) for b in blocks]
    nb = len(blocks)
    bm_all = vsa_map_from_lists(kv_list, kv_num, nb, npre, w.topk, sizes)
    ref = _vsa_check_map(bm_all[heads], q, k, blocks, npre, w.topk, w.scale, heads)
    rng = np.random.default_rng(16)
    sample = [0, npre, nb - 1] + [int(x) for x in rng.integers(npre, nb, 4)]
    out_h, lse_h = to_np(out), to_np(lse)
    checked = 0
    for x, h in enumerate(heads):
        for i in sample:
            if not np.array_equal(bm_all[h, i], ref[x, i]):
                continue  # a near-tie resolved the other way; the map check covered it
            rows = torch.from_numpy(blocks[i])
            keys = torch.from_numpy(np.concatenate([blocks[j] for j in np.nonzero(ref[x, i])[0]]))
            r_o, r_l = oracle.attention_single(q[rows, h:h + 1], k[keys, h:h + 1], v[keys, h:h + 1], w.scale, False)
            assert_close(out_h[blocks[i], h:h + 1], lse_h[h:h + 1, blocks[i]], r_o, r_l, what=f"head {h} block {i}")
            checked += 1
    assert checked >= len(sample)
