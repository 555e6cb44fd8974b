"""attn_fwd_paged_noalloc, the paged decode for callers that cannot allocate
device memory while it runs (a CUDA-graph capture, a framework plugin with no
allocator, a server with a fixed memory budget).  It must give what the
workspace entry point attn_fwd_paged gives, call after call, although every
call reuses the same built-in scratch.

This file is named so that pytest collects it last."""

import ctypes

import numpy as np
import pytest
import torch

import attention_forward_09_gb300 as gb
import oracle
import workloads
from _helpers import LSE_TOL, OUT_TOL, max_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from attention_forward_09_gb300 import _build

    _build.build()
    return gb.load_library()


def _inputs(w):
    dev = torch.device("cuda:0")
    q, cache, bt, sl = w.make()
    return q.to(dev), cache.to(dev), bt.to(dev), sl.to(dev)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(lib):
    w = workloads.Paged("noalloc", [300, 1, 2500, 129, 4096], 16, 4, 128, seed=21)
    q, cache, bt, sl = _inputs(w)
    ora_out, ora_lse = oracle.attention_paged(*w.make(), w.scale)  # the float64 oracle on the same inputs
    max_len = max(w.seq_lens)
    ref_out, ref_lse = gb.attn_fwd_paged(q, cache, bt, sl, max_len, w.scale, lse=True)
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        # through the C ABI directly, with preallocated outputs: nothing is allocated for the call
        st = lib.attn_fwd_paged_noalloc(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(cache.data_ptr()), cache.shape[1], 128,
            ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(sl.data_ptr()), q.shape[0], max_len,
            w.Hq, w.Hkv, w.D, w.scale, 1, ctypes.c_void_p(out.data_ptr()), gb.OUT_F32,
            ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(status.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        assert st == 0 and int(status.item()) == 0
        assert max_err(to_np(out), to_np(ref_out)) <= OUT_TOL
        assert max_err(to_np(lse), to_np(ref_lse)) <= LSE_TOL
        assert max_err(to_np(out), ora_out) <= OUT_TOL
        assert max_err(to_np(lse), ora_lse) <= LSE_TOL


def test_noalloc_binding_and_size_limit(lib):
    w = workloads.Paged("noalloc_b", [700, 64], 8, 8, 64, seed=4)
    q, cache, bt, sl = _inputs(w)
    a, la = gb.attn_fwd_paged(q, cache, bt, sl, max(w.seq_lens), w.scale, lse=True)
    b, lb = gb.attn_fwd_paged_noalloc(q, cache, bt, sl, max(w.seq_lens), w.scale, lse=True)
    torch.cuda.synchronize()
    assert max_err(to_np(b), to_np(a)) <= OUT_TOL and max_err(to_np(lb), to_np(la)) <= LSE_TOL
    ro, rl = oracle.attention_paged(*w.make(), w.scale)
    assert max_err(to_np(b), ro) <= OUT_TOL and max_err(to_np(lb), rl) <= LSE_TOL
    with pytest.raises(gb.GbattnError) as e:  # more sequences than the scratch can hold partials for
        gb.attn_fwd_paged_noalloc(q[:1].expand(4096, -1, -1).contiguous(), cache, bt[:1].expand(4096, -1).contiguous(),
                                  sl[:1].expand(4096).contiguous(), 131072, w.scale)
    assert e.value.status == 7
