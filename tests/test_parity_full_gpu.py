"""Whole-workload parity at the full sizes the bench times: every output
element and every LSE element of each workload, computed by the library in
the bench's launch configuration (fp32 out + lse through the same entry
point), is compared with the float64 oracle (max |out err| <= 1e-2, max |lse
err| <= 1e-3).  The oracle runs once per (document or batch entry, head) on
the host cores, in a spawn process pool.

Workloads: diffusion-transformer self-attention (B=2, S=4096, 24 heads,
D=128); packed causal prefill with GQA (8 documents, 32/8 heads, D=128);
paged decode (64 sequences, 32/8 heads, D=128, contexts up to 32768);
cross-attention (16384 video queries x 512 text keys, 40 heads); dense
self-attention at S=8192, 16 heads, D in {64, 96, 192, 256}."""

import math

import numpy as np
import pytest
import torch

import attention_forward_09_gb300 as gb
import oracle
import workloads
from _helpers import LSE_TOL, OUT_TOL, dev, max_err, status_word
from _oracle_pool import f32, run_units, score_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_09_gb300 import _build

    _build.build()
    gb.load_library()


def _compare_units(units, got, what):
    """units: [(key, q, k, v, scale, causal)], got[key] = (out [L, D] fp32 numpy,
    lse [L] fp32 numpy).  Returns the worst errors; fails on the first unit
    beyond tolerance."""
    res = run_units([u[1:] for u in units], max(score_bytes(u[1].shape[0], u[2].shape[0]) for u in units))
    worst_o = worst_l = 0.0
    for u, (ro, rl) in zip(units, res):
        go, gl = got(u[0])
        eo = max_err(go, ro[:, 0])
        el = max_err(gl, rl[0])
        assert eo <= OUT_TOL, f"{what} unit {u[0]}: max |out err| {eo:.3e}"
        assert el <= LSE_TOL, f"{what} unit {u[0]}: max |lse err| {el:.3e}"
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
    return worst_o, worst_l


def _full_dense(w):
    q, k, v = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_dense(q.to(dev()), k.to(dev()), v.to(dev()), w.scale, w.causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert out.dtype == torch.float32
    out_h, lse_h = out.cpu().numpy(), lse.cpu().numpy()
    del out, lse
    g = w.Hq // w.Hkv
    units = [((b, h), f32(q[b, :, h:h + 1]), f32(k[b, :, h // g:h // g + 1]), f32(v[b, :, h // g:h // g + 1]),
              w.scale, w.causal) for b in range(w.B) for h in range(w.Hq)]
    return _compare_units(units, lambda key: (out_h[key[0], :, key[1]], lse_h[key[0], key[1]]), w.name)


def test_full_dit_self_attention():
    _full_dense(workloads.dit_self())


def test_full_cross_attention():
    _full_dense(workloads.cross_attn())


@pytest.mark.parametrize("D", [64, 96, 192, 256])
def test_full_head_sweep(D):
    _full_dense(workloads.head_sweep(D))


def test_full_varlen_causal_gqa():
    w = workloads.varlen_causal_gqa()
    q, k, v, cq, ck = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_varlen(q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()),
                                  max(w.lens_q), max(w.lens_k), w.scale, w.causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out_h, lse_h = out.cpu().numpy(), lse.cpu().numpy()
    g = w.Hq // w.Hkv
    units = []
    for n in range(len(w.lens_q)):
        a, b, c, d = int(cq[n]), int(cq[n + 1]), int(ck[n]), int(ck[n + 1])
        for h in range(w.Hq):
            units.append(((a, b, h), f32(q[a:b, h:h + 1]), f32(k[c:d, h // g:h // g + 1]),
                          f32(v[c:d, h // g:h // g + 1]), w.scale, w.causal))
    _compare_units(units, lambda key: (out_h[key[0]:key[1], key[2]], lse_h[key[2], key[0]:key[1]]), w.name)


def test_full_paged_decode():
    w = workloads.paged_decode()
    q, cache, bt, sl = w.make(chunk_rows=256)
    st = status_word()
    out, lse = gb.attn_fwd_paged(q.to(dev()), cache.to(dev()), bt.to(dev()), sl.to(dev()), max(w.seq_lens),
                                 w.scale, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out_h, lse_h = out.cpu().numpy(), lse.cpu().numpy()
    # every sequence, eight at a time (the oracle's gather holds float64 K/V of the sequences it is given)
    for s0 in range(0, len(w.seq_lens), 8):
        s1 = min(len(w.seq_lens), s0 + 8)
        ro, rl = oracle.attention_paged(q[s0:s1], cache, bt[s0:s1], sl[s0:s1], w.scale)
        eo, el = max_err(out_h[s0:s1], ro), max_err(lse_h[s0:s1], rl)
        assert eo <= OUT_TOL and el <= LSE_TOL, f"sequences {s0}..{s1 - 1}: out {eo:.3e}, lse {el:.3e}"


def test_full_tiny_varlen():
    w = workloads.tiny_varlen()
    q, k, v, cq, ck = w.make()
    st = status_word()
    out, lse = gb.attn_fwd_varlen(q.to(dev()), k.to(dev()), v.to(dev()), cq.to(dev()), ck.to(dev()),
                                  max(w.lens_q), max(w.lens_k), w.scale, w.causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle.attention_varlen(q, k, v, cq, ck, w.scale, w.causal)
    assert max_err(out.cpu().numpy(), ro) <= OUT_TOL
    assert max_err(lse.cpu().numpy(), rl) <= LSE_TOL
    assert math.isclose(w.scale, 1.0 / 8.0)
