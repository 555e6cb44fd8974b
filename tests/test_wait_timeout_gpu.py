"""A pipeline wait that runs out: the kernel sets GBATTN_DEV_TIMEOUT, lets
its copies land, frees its tensor memory and returns; the call comes back
and the context stays usable (a following normal call matches the oracle
with a clean status).  For the duration of one call the kernels are told to
give up their waits at once (attn_set_wait_give_up): no fault is planted and
nothing is left waiting.

The launches are the one-tile kernel (D = 256) and a causal two-tile launch
(D = 64, 128) of a single CTA: no cluster, no persistent grid."""

import math

import pytest
import torch

import attention_forward_09_gb300 as gb
import oracle
import workloads
from _helpers import assert_close, dev, status_word

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_09_gb300 import _build

    _build.build()
    gb.load_library()


@pytest.mark.parametrize("D,Sq,causal", [(256, 128, False), (128, 256, True), (64, 256, True)])
def test_wait_that_gives_up_reports_timeout_and_the_context_stays_usable(D, Sq, causal):
    Sk = 2048
    if not causal:
        assert gb.attn_fwd_dense_plan(1, Sq, Sk, 1, 1, D, causal) == (1, 0)
    g = torch.Generator().manual_seed(D)
    q, k, v = (workloads.randn_bf16(g, 1, n, 1, D).to(dev()) for n in (Sq, Sk, Sk))
    s = 1.0 / math.sqrt(D)
    prev = gb.attn_set_wait_give_up(True)
    try:
        st = status_word()
        gb.attn_fwd_dense(q, k, v, s, causal, lse=True, dev_status=st)
        torch.cuda.synchronize()  # the call comes back
        assert int(st.item()) & gb.DEV_TIMEOUT
    finally:
        gb.attn_set_wait_give_up(prev)
    st = status_word()
    out, lse = gb.attn_fwd_dense(q, k, v, s, causal, lse=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle.attention_dense(q.cpu(), k.cpu(), v.cpu(), s, causal)
    assert_close(out, lse, ro, rl, what=f"after a timed-out call, D={D}")
