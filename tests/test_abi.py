"""The C-ABI library builds, loads, exports every declared symbol, and rejects
bad arguments on the host before touching the GPU (these calls make no CUDA
call, so they run on a machine without a GPU)."""

import ctypes
import json
import os
import re

import pytest

import attention_forward_09_gb300 as gb
from attention_forward_09_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gb.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(
        ["attn_fwd_dense", "attn_fwd_varlen", "attn_fwd_paged", "attn_fwd_paged_workspace_size",
         "attn_status_string", "attn_fwd_paged_noalloc", "attn_fwd_dense_plan", "attn_fwd_varlen_plan",
         "attn_set_wait_give_up", "attn_fwd_padded",
         "attn_kv_cache_write",
         "attn_fwd_paged_prefill", "attn_mask_to_varlen", "attn_pack_rows", "attn_unpack_rows",
         "attn_unpack_lse", "attn_vsa_layout", "attn_vsa_tile_map", "attn_gather_rows", "attn_vsa_pool",
         "attn_vsa_list_size", "attn_vsa_block_map", "attn_fwd_vsa"])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in gb.SIGNATURES, name


def test_status_strings(lib):
    for code in range(8):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(99) == b"unknown status"


# A fake, 16-byte aligned "device" address: validation must fail before any use.
P = ctypes.c_void_p(0x10000)
UNALIGNED = ctypes.c_void_p(0x10008)


def dense(lib, **kw):
    a = dict(q=P, k=P, v=P, B=1, Sq=8, Sk=8, Hq=4, Hkv=2, D=128, scale=0.1, causal=0, out=P, odt=1, lse=None)
    a.update(kw)
    return lib.attn_fwd_dense(a["q"], a["k"], a["v"], a["B"], a["Sq"], a["Sk"], a["Hq"], a["Hkv"], a["D"],
                              a["scale"], a["causal"], a["out"], a["odt"], a["lse"], None, None)


def test_dense_validation(lib):
    assert dense(lib, D=80) == UNSUPPORTED
    assert dense(lib, D=32) == UNSUPPORTED
    assert dense(lib, Hq=6, Hkv=4) == INVALID
    assert dense(lib, Hkv=0) == INVALID
    assert dense(lib, q=None) == INVALID
    assert dense(lib, out=None) == INVALID
    assert dense(lib, scale=0.0) == INVALID
    assert dense(lib, scale=-1.0) == INVALID
    assert dense(lib, scale=float("nan")) == INVALID
    assert dense(lib, odt=7) == UNSUPPORTED
    assert dense(lib, k=UNALIGNED) == ALIGN
    assert dense(lib, B=-1) == INVALID
    # empty problems are a no-op success without touching the device
    assert dense(lib, B=0) == OK
    assert dense(lib, Sq=0) == OK


def varlen(lib, **kw):
    a = dict(cq=P, ck=P, N=2, Tq=16, Tk=16, mq=8, mk=8, Hq=4, Hkv=4, D=64, out=P)
    a.update(kw)
    return lib.attn_fwd_varlen(P, P, P, a["cq"], a["ck"], a["N"], a["Tq"], a["Tk"], a["mq"], a["mk"], a["Hq"],
                               a["Hkv"], a["D"], 0.125, 0, a["out"], 1, None, None, None)


def test_varlen_validation(lib):
    assert varlen(lib, cq=None) == INVALID
    assert varlen(lib, ck=None) == INVALID
    assert varlen(lib, mq=17) == INVALID  # a document cannot be longer than the tensor
    assert varlen(lib, N=-1) == INVALID
    assert varlen(lib, D=100) == UNSUPPORTED
    assert varlen(lib, N=0) == OK
    assert varlen(lib, Tq=0, mq=0) == OK


def paged(lib, **kw):
    a = dict(nb=16, bs=128, bt=P, maxb=4, sl=P, S=2, maxlen=512, Hq=8, Hkv=2, D=128, ws=P, wsb=1 << 30)
    a.update(kw)
    return lib.attn_fwd_paged(P, P, a["nb"], a["bs"], a["bt"], a["maxb"], a["sl"], a["S"], a["maxlen"], a["Hq"],
                              a["Hkv"], a["D"], 0.1, 1, P, 1, None, a["ws"], a["wsb"], None, None)


def test_paged_validation(lib):
    assert paged(lib, bs=64) == UNSUPPORTED  # AscendAttentionBackend.get_supported_block_size is [128]
    assert paged(lib, bt=None) == INVALID
    assert paged(lib, sl=None) == INVALID
    assert paged(lib, Hq=6, Hkv=4) == INVALID
    assert paged(lib, D=48) == UNSUPPORTED
    assert paged(lib, ws=None) == WORKSPACE
    assert paged(lib, wsb=16) == WORKSPACE
    assert paged(lib, ws=ctypes.c_void_p(0x10010)) == WORKSPACE  # must be 256-byte aligned
    assert paged(lib, S=0) == OK


def test_workspace_size_is_pure_and_sized_for_the_plan(lib):
    f = lib.attn_fwd_paged_workspace_size
    a = f(64, 32, 8, 128, 32768)
    assert a == f(64, 32, 8, 128, 32768) and a > 0
    # one partial (D floats + 1 lse float) per (seq, q head, split)
    assert a >= 64 * 32 * (128 + 1) * 4
    assert f(64, 32, 8, 80, 32768) == 0 and f(0, 32, 8, 128, 100) == 0 and f(4, 6, 4, 128, 100) == 0
    assert f(1, 8, 8, 128, 1) > 0


def test_noalloc_refuses_sizes_beyond_its_scratch_on_the_host(lib):
    """The size check comes before any CUDA call, so it runs without a GPU."""
    S, Hq, Hkv, D, L = 4096, 64, 8, 256, 131072
    assert lib.attn_fwd_paged_workspace_size(S, Hq, Hkv, D, L) > gb.NOALLOC_SCRATCH_BYTES
    st = lib.attn_fwd_paged_noalloc(P, P, 1 << 20, 128, P, L // 128, P, S, L, Hq, Hkv, D, 0.1, 1, P, 1, None,
                                    None, None)
    assert st == 7


def test_dense_plan_validates_before_touching_a_device(lib):
    n, sp = ctypes.c_int(7), ctypes.c_int(7)
    assert lib.attn_fwd_dense_plan(1, 8, 8, 4, 3, 128, 0, ctypes.byref(n), ctypes.byref(sp)) == 1  # Hq % Hkv
    assert (n.value, sp.value) == (0, 0)
    assert lib.attn_fwd_dense_plan(1, 8, 8, 4, 2, 80, 0, ctypes.byref(n), ctypes.byref(sp)) == 2  # head size
    assert lib.attn_fwd_dense_plan(1, 8, 8, 4, 2, 128, 0, None, ctypes.byref(sp)) == 1
    assert lib.attn_fwd_dense_plan(0, 8, 8, 4, 2, 128, 0, ctypes.byref(n), ctypes.byref(sp)) == 0  # nothing to do
    assert (n.value, sp.value) == (0, 0)


def test_kv_cache_write_validates_before_touching_a_device(lib):
    w = lib.attn_kv_cache_write
    assert w(P, P, P, -1, P, 8, 128, 8, 128, None, None) == 1          # negative token count
    assert w(P, P, P, 4, P, 0, 128, 8, 128, None, None) == 1           # no blocks
    assert w(P, P, P, 4, P, 8, 0, 8, 128, None, None) == 1             # block size
    assert w(P, P, P, 4, P, 8, 128, 8, 80, None, None) == 2            # head size
    assert w(None, P, P, 4, P, 8, 128, 8, 128, None, None) == 1        # null key
    assert w(UNALIGNED, P, P, 4, P, 8, 128, 8, 128, None, None) == 3   # alignment
    assert w(P, P, P, 0, P, 8, 128, 8, 128, None, None) == 0           # nothing to write
    assert w(P, P, P, 1 << 30, P, 8, 128, 8, 128, None, None) == 2     # row count past 32 bits
    assert w(P, P, P, 4, P, 8, 128, 1 << 22, 256, None, None) == 2     # row bytes past 32 bits


def test_paged_prefill_validates_before_touching_a_device(lib):
    def call(**kw):
        a = dict(q=P, c=P, nb=8, bs=128, bt=P, mb=4, sl=P, cu=P, S=2, Tq=10, mq=5, ml=300, Hq=4, Hkv=2, D=128,
                 scale=0.1, causal=1, out=P, odt=1, lse=None)
        a.update(kw)
        return lib.attn_fwd_paged_prefill(a["q"], a["c"], a["nb"], a["bs"], a["bt"], a["mb"], a["sl"], a["cu"],
                                          a["S"], a["Tq"], a["mq"], a["ml"], a["Hq"], a["Hkv"], a["D"], a["scale"],
                                          a["causal"], a["out"], a["odt"], a["lse"], None, None)
    assert call(bs=64) == 2           # block size
    assert call(D=80) == 2            # head size
    assert call(Hkv=3) == 1           # Hq % Hkv
    assert call(cu=None) == 1         # missing cu_seqlens_q
    assert call(mq=11) == 1           # max_seqlen_q > Tq
    assert call(q=UNALIGNED) == 3     # alignment
    assert call(S=0) == 0             # nothing to compute


def test_mask_helpers_validate_before_touching_a_device(lib):
    assert lib.attn_mask_to_varlen(P, -1, 8, P, P, None) == 1
    assert lib.attn_mask_to_varlen(None, 2, 8, P, P, None) == 1
    assert lib.attn_mask_to_varlen(P, 0, 8, P, P, None) == 0
    assert lib.attn_pack_rows(P, P, P, 2, 8, 24, P, None) == 1          # row bytes not a multiple of 16
    assert lib.attn_pack_rows(UNALIGNED, P, P, 2, 8, 256, P, None) == 3
    assert lib.attn_unpack_rows(P, P, 2, 8, 256, UNALIGNED, None) == 3
    assert lib.attn_unpack_lse(P, P, 2, 0, 8, P, None) == 1             # no heads
    assert lib.attn_pack_rows(P, P, P, 1 << 16, 1 << 16, 256, P, None) == 2  # B * S >= 2^31


def test_dense_refuses_row_counts_past_32_bits(lib):
    assert dense(lib, B=65535, Sq=40000) == 2
    assert dense(lib, B=65535, Sq=8, Sk=40000) == 2


@pytest.mark.parametrize("prefix,shape", [([70, 5], (5, 6, 7)), ([], (4, 4, 6)), ([128], (1, 1, 1)), ([3], (9, 2, 13))])
def test_vsa_layout_equals_the_oracle_blocks(lib, prefix, shape):
    """A host computation: runs without a GPU, bit-exact against the oracle."""
    import oracle
    order, start, npre = gb.attn_vsa_layout(prefix, shape)
    blocks, n_prefix = oracle.vsa_blocks(prefix, shape)
    assert npre == n_prefix and start.numel() == len(blocks) + 1
    for b, ref in enumerate(blocks):
        assert order[int(start[b]):int(start[b + 1])].tolist() == ref.tolist()


def _vsa_layout_cases():
    with open(os.path.join(ROOT, "tests", "golden", "vsa_layout_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _vsa_layout_cases(), ids=lambda c: c["name"])
def test_vsa_host_layouts_match_the_hand_worked_layouts(lib, case):
    """Both host layout calls against block layouts worked by hand from the
    page's tiling functions (no oracle involved)."""
    blocks = [[i for a, b in runs for i in range(a, b)] for runs in case["blocks"]]
    order, start, npre = gb.attn_vsa_layout(case["prefix"], case["video"])
    assert npre == case["n_prefix_blocks"]
    assert [order[int(start[b]):int(start[b + 1])].tolist() for b in range(len(blocks))] == blocks
    assert start.numel() == len(blocks) + 1
    index, sizes, npre = gb.attn_vsa_tile_map(case["prefix"], case["video"])
    assert npre == case["n_prefix_blocks"] and sizes.tolist() == case["block_sizes"]
    nb = len(blocks)
    expect = [-1] * ((nb + nb % 2) * 64)
    for b, toks in enumerate(blocks):
        expect[64 * b:64 * b + len(toks)] = toks
    assert index.tolist() == expect


def test_vsa_layout_validation(lib):
    nb, npre = ctypes.c_int(), ctypes.c_int()
    seg = (ctypes.c_int32 * 1)(-1)
    assert lib.attn_vsa_layout(seg, 1, 4, 4, 4, 4, 4, 4, 64, None, None, ctypes.byref(nb), ctypes.byref(npre)) == 1
    assert lib.attn_vsa_layout(None, 0, 4, 4, 4, 8, 4, 4, 64, None, None, ctypes.byref(nb), ctypes.byref(npre)) == 1


@pytest.mark.parametrize("prefix,shape", [([100, 37], (5, 9, 10)), ([], (8, 12, 12)), ([3], (9, 2, 13))])
def test_vsa_tile_map_equals_the_oracle_blocks(lib, prefix, shape):
    """Host computation: tiled row 64 b + r holds token r of block b, -1 past
    the block's end and in the empty partner of an odd block count."""
    import oracle
    index, sizes, npre = gb.attn_vsa_tile_map(prefix, shape)
    blocks, n_prefix = oracle.vsa_blocks(prefix, shape)
    nb = len(blocks)
    assert npre == n_prefix and sizes.tolist() == [len(b) for b in blocks]
    assert index.numel() == (nb + nb % 2) * 64
    for b, ref in enumerate(blocks):
        assert index[64 * b:64 * b + len(ref)].tolist() == ref.tolist()
        assert (index[64 * b + len(ref):64 * b + 64] == -1).all()
    assert (index[64 * nb:] == -1).all()


def test_vsa_list_size_counts_the_tiles(lib):
    # 21 blocks, 3 prefix, topk 5: tiles 0-1 list all 21 blocks, tiles 2-10 at most 3 + 2 * 5
    assert gb.attn_vsa_list_size(21, 3, 5, 1) == 2 * 21 + 9 * 13
    assert gb.attn_vsa_list_size(21, 3, 5, 4) == 4 * (2 * 21 + 9 * 13)
    assert gb.attn_vsa_list_size(18, 0, 7, 1) == 9 * 14
    assert gb.attn_vsa_list_size(5, 1, 100, 2) == 2 * 3 * 5      # every block kept: every tile lists all
    n = ctypes.c_longlong()
    assert lib.attn_vsa_list_size(21, 3, 0, 1, ctypes.byref(n)) == 1  # topk must be positive
    assert lib.attn_vsa_list_size(21, 22, 5, 1, ctypes.byref(n)) == 1


def test_vsa_device_calls_validate_before_touching_a_device(lib):
    assert lib.attn_gather_rows(P, 10, P, 10, 24, P, None, None) == 1           # row bytes not a multiple of 16
    assert lib.attn_gather_rows(UNALIGNED, 10, P, 10, 256, P, None, None) == 3
    assert lib.attn_gather_rows(P, 10, P, 0, 256, P, None, None) == 0           # nothing to copy
    assert lib.attn_vsa_pool(P, 4, 2, 80, P, P, None, None) == 2                # head size
    assert lib.attn_vsa_pool(P, 4, 2, 128, P, UNALIGNED, None, None) == 3
    assert lib.attn_vsa_block_map(P, P, 21, 3, 4, 3, 128, 5, 0.1, P, P, P, None, None) == 1  # Hq % Hkv
    assert lib.attn_vsa_block_map(P, P, 21, 3, 4, 2, 128, 0, 0.1, P, P, P, None, None) == 1  # topk 0
    assert lib.attn_vsa_block_map(P, P, 30000, 0, 4, 2, 256, 5, 0.1, P, P, P, None, None) == 2  # scores too big
    assert lib.attn_vsa_block_map(UNALIGNED, P, 21, 3, 4, 2, 128, 5, 0.1, P, P, P, None, None) == 3
    assert lib.attn_vsa_block_map(P, UNALIGNED, 21, 3, 4, 2, 128, 5, 0.1, P, P, P, None, None) == 3

    def fwd(**kw):
        a = dict(q=P, k=P, v=P, nb=21, npre=3, topk=5, kl=P, kn=P, idx=P, rows=587, hq=4, hkv=2, d=128,
                 scale=0.1, out=P, odt=1, lse=None)
        a.update(kw)
        return lib.attn_fwd_vsa(a["q"], a["k"], a["v"], a["nb"], a["npre"], a["topk"], a["kl"], a["kn"], a["idx"],
                                a["rows"], a["hq"], a["hkv"], a["d"], a["scale"], a["out"], a["odt"], a["lse"],
                                None, None)
    assert fwd(d=96) == 2                # the attention kernel serves D = 64 and 128
    assert fwd(odt=7) == 2
    assert fwd(idx=None) == 1            # a tiled output needs out_rows = nbp * 64
    assert fwd(idx=None, rows=22 * 64, nb=0, npre=0) == 1
    assert fwd(nb=0, npre=0, rows=0) == 0  # nothing to compute
    assert fwd(k=UNALIGNED) == 3
    assert fwd(nb=200000) == 2           # more than 65535 tiles
    assert fwd(scale=-1.0) == 1


# The binding checks every tensor size the C calls of block-sparse video
# attention derive from their integer arguments, before any device check, so
# a mismatched tensor is refused on the host (CPU tensors suffice here).

def _vsa_fwd_args(nb=21, npre=3, topk=5, hq=4, hkv=2, d=128):
    import torch

    rows = (nb + nb % 2) * 64
    q = torch.zeros(rows, hq, d, dtype=torch.bfloat16)
    kv = torch.zeros(rows, hkv, d, dtype=torch.bfloat16)
    kl = torch.zeros(gb.attn_vsa_list_size(nb, npre, topk, hq), dtype=torch.int32)
    kn = torch.zeros(hq, (nb + 1) // 2, dtype=torch.int32)
    idx = torch.zeros(rows, dtype=torch.int32)
    return dict(q_tiled=q, k_tiled=kv, v_tiled=kv.clone(), kv_list=kl, kv_num=kn, num_blocks=nb,
                num_prefix_blocks=npre, topk=topk, out_index=idx, out_rows=1000)


@pytest.mark.parametrize("change,message", [
    (lambda a: a.update(q_tiled=a["q_tiled"][:-64]), "rows"),
    (lambda a: a.update(k_tiled=a["k_tiled"][:-1]), "k_tiled and v_tiled"),
    (lambda a: a.update(v_tiled=a["v_tiled"][..., :64].contiguous()), "k_tiled and v_tiled"),
    (lambda a: a.update(kv_list=a["kv_list"][:-1]), "kv_list holds"),
    (lambda a: a.update(kv_list=a["kv_list"].long()), "kv_list must be"),
    (lambda a: a.update(kv_num=a["kv_num"][:, :-1].contiguous()), "kv_num must be"),
    (lambda a: a.update(out_index=a["out_index"][:-1]), "out_index"),
    (lambda a: a.update(out_index=None), "out_rows must equal"),
    (lambda a: a.update(out=__import__("torch").zeros(999, 4, 128)), "out must be"),
    (lambda a: a.update(lse=__import__("torch").zeros(4, 999)), "lse must be"),
])
def test_vsa_fwd_binding_refuses_mismatched_tensors(lib, change, message):
    a = _vsa_fwd_args()
    change(a)
    with pytest.raises(ValueError, match=message):
        gb.attn_fwd_vsa(**a)


def test_vsa_fwd_binding_shape_check_accepts_matching_tensors(lib):
    a = _vsa_fwd_args()
    with pytest.raises(ValueError, match="CUDA"):  # past the size checks, stopped by the device check
        gb.attn_fwd_vsa(**a)


def test_vsa_block_map_binding_refuses_mismatched_tensors(lib):
    import torch

    pq, pk = torch.zeros(4, 21, 128), torch.zeros(2, 21, 128)
    sizes = torch.full((21,), 64, dtype=torch.int32)
    with pytest.raises(ValueError, match="same nb and D"):
        gb.attn_vsa_block_map(pq, torch.zeros(2, 20, 128), sizes, 3, 5, 0.1)
    with pytest.raises(ValueError, match="same nb and D"):
        gb.attn_vsa_block_map(pq, torch.zeros(2, 21, 64), sizes, 3, 5, 0.1)
    with pytest.raises(ValueError, match="float32"):
        gb.attn_vsa_block_map(pq.double(), pk, sizes, 3, 5, 0.1)
    with pytest.raises(ValueError, match="block_sizes"):
        gb.attn_vsa_block_map(pq, pk, sizes[:-1], 3, 5, 0.1)


def test_varlen_plan_validates_before_touching_a_device(lib):
    n = ctypes.c_int(7)
    assert lib.attn_fwd_varlen_plan(8, 1000, 200, 200, 32, 8, 80, 1, ctypes.byref(n)) == UNSUPPORTED
    assert lib.attn_fwd_varlen_plan(8, 1000, 200, 200, 6, 4, 128, 1, ctypes.byref(n)) == INVALID
    assert lib.attn_fwd_varlen_plan(8, 1000, 200, 200, 32, 8, 128, 1, None) == INVALID
    assert lib.attn_fwd_varlen_plan(0, 0, 0, 0, 32, 8, 128, 1, ctypes.byref(n)) == OK and n.value == 0


def test_wait_give_up_switch_is_host_only_and_restores(lib):
    prev = ctypes.c_int(-5)
    assert lib.attn_set_wait_give_up(2, ctypes.byref(prev)) == INVALID
    assert lib.attn_set_wait_give_up(1, ctypes.byref(prev)) == OK and prev.value == 0
    assert gb.attn_set_wait_give_up(False) is True
    assert gb.attn_set_wait_give_up(False) is False


def test_padded_validation(lib):
    def padded(**kw):
        a = dict(q=P, k=P, v=P, lq=None, lk=P, B=2, Sq=8, Sk=8, Hq=4, Hkv=2, D=128, scale=0.1, causal=0, out=P,
                 odt=1, lse=None)
        a.update(kw)
        return lib.attn_fwd_padded(a["q"], a["k"], a["v"], a["lq"], a["lk"], a["B"], a["Sq"], a["Sk"], a["Hq"],
                                   a["Hkv"], a["D"], a["scale"], a["causal"], a["out"], a["odt"], a["lse"], None,
                                   None)
    assert padded(D=80) == UNSUPPORTED
    assert padded(Hq=6, Hkv=4) == INVALID
    assert padded(q=None) == INVALID
    assert padded(scale=0.0) == INVALID
    assert padded(v=UNALIGNED) == ALIGN
    assert padded(B=-1) == INVALID
    assert padded(B=70000) == UNSUPPORTED
    assert padded(B=0) == OK  # nothing to compute, no device touched
