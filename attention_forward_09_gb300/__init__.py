"""GB300 (sm_103a) fused attention forward -- Python binding of libgbattn.so.

The functions here only marshal arguments (shapes, pointers, the current
CUDA stream) into the C ABI declared in ``include/gbattn.h``; every step of
the computation runs in the library's CUDA kernels.  There is no CPU or
PyTorch fallback: if the library is missing, or the device is not a GB300,
the calls raise.

Entry points (same names as the C ABI):
    attn_fwd_dense(q, k, v, ...)    q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D]
    attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, ...)
    attn_fwd_paged(q, kv_cache, block_table, seq_lens, max_seq_len, ...)
    attn_fwd_paged_workspace_size(num_seqs, Hq, Hkv, D, max_seq_len)
    attn_kv_cache_write, attn_fwd_paged_prefill, attn_mask_to_varlen, attn_pack_rows,
    attn_unpack_rows, attn_unpack_lse, attn_fwd_dense_plan, attn_fwd_varlen_plan, attn_fwd_paged_noalloc,
    attn_set_wait_give_up, attn_fwd_padded
    attn_vsa_layout, attn_vsa_tile_map, attn_gather_rows, attn_vsa_pool, attn_vsa_list_size,
    attn_vsa_block_map, attn_fwd_vsa
Compositions of those calls: attn_fwd_masked (padding mask), attn_vsa (block-sparse
video attention, with VsaPlan holding one geometry's layout on the device).
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbattn.so")

OUT_BF16, OUT_F32 = 0, 1
DEV_BAD_INDEX, DEV_TIMEOUT, DEV_BAD_SEQLEN = 1, 2, 4
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "alignment", 4: "workspace",
                5: "cuda", 6: "device", 7: "scratch limit"}
NOALLOC_SCRATCH_BYTES = 32 << 20  # GBATTN_NOALLOC_SCRATCH_BYTES

# (name, restype, argtypes) for every symbol of include/gbattn.h
_P, _I, _F, _Z, _L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong
SIGNATURES = {
    "attn_fwd_dense": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P, _P, _P]),
    "attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P, _P, _P]),
    "attn_fwd_paged_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attn_fwd_paged": (_I, [_P, _P, _I, _I, _P, _I, _P, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P, _P, _Z, _P, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_fwd_paged_noalloc": (_I, [_P, _P, _I, _I, _P, _I, _P, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P, _P, _P]),
    "attn_fwd_dense_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "attn_fwd_varlen_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "attn_fwd_padded": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P, _P, _P]),
    "attn_set_wait_give_up": (_I, [_I, ctypes.POINTER(ctypes.c_int)]),
    "attn_kv_cache_write": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P]),
    "attn_fwd_paged_prefill": (_I, [_P, _P, _I, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _I, _P,
                                    _P, _P]),
    "attn_mask_to_varlen": (_I, [_P, _I, _I, _P, _P, _P]),
    "attn_pack_rows": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "attn_unpack_rows": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "attn_unpack_lse": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "attn_vsa_layout": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.POINTER(ctypes.c_int),
                             ctypes.POINTER(ctypes.c_int)]),
    "attn_vsa_tile_map": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.POINTER(ctypes.c_int),
                               ctypes.POINTER(ctypes.c_int)]),
    "attn_gather_rows": (_I, [_P, _L, _P, _L, _I, _P, _P, _P]),
    "attn_vsa_pool": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "attn_vsa_list_size": (_I, [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_longlong)]),
    "attn_vsa_block_map": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "attn_fwd_vsa": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _L, _I, _I, _I, _F, _P, _I, _P, _P, _P]),
}

_lib = None


class GbattnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({STATUS_NAMES.get(status, '?')})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgbattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with attention_forward_09_gb300._build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, st):
    if st != 0:
        raise GbattnError(fn, st)


def _out_code(dtype):
    if dtype == torch.float32:
        return OUT_F32
    if dtype == torch.bfloat16:
        return OUT_BF16
    raise ValueError("out dtype must be float32 or bfloat16")


def _bf16_cuda(name, t):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")


def attn_fwd_dense(q, k, v, softmax_scale=None, causal=False, out=None, lse=None, out_dtype=torch.float32,
                   dev_status=None, stream=None):
    """Dense batch.  Returns (out [B, Sq, Hq, D], lse [B, Hq, Sq] or None).
    Pass ``lse=True`` to allocate the LSE output, or a float32 tensor."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Sk, Hkv, D] matching q")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty(B, Sq, Hq, D, dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    st = load_library().attn_fwd_dense(_ptr(q), _ptr(k), _ptr(v), B, Sq, Sk, Hq, Hkv, D, scale, int(bool(causal)),
                                       _ptr(out), _out_code(out.dtype), _ptr(lse), _ptr(dev_status),
                                       _stream_handle(stream))
    _check("attn_fwd_dense", st)
    return out, lse


def attn_fwd_padded(q, k, v, lens_q=None, lens_k=None, softmax_scale=None, causal=False, out=None, lse=None,
                    out_dtype=torch.float32, dev_status=None, stream=None):
    """Right-padded batch: entry b uses its first lens_q[b] query rows and
    lens_k[b] keys (int32 CUDA tensors [B], or None for all rows).  q [B, Sq,
    Hq, D], k/v [B, Sk, Hkv, D].  Returns (out [B, Sq, Hq, D], lse [B, Hq, Sq]
    or None); padded query rows get zeros and -inf."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Sk, Hkv, D] matching q")
    for n, t in (("lens_q", lens_q), ("lens_k", lens_k)):
        if t is not None and (t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.numel() != B):
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor of {B} entries")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty(B, Sq, Hq, D, dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    st = load_library().attn_fwd_padded(_ptr(q), _ptr(k), _ptr(v), _ptr(lens_q), _ptr(lens_k), B, Sq, Sk, Hq, Hkv, D,
                                        scale, int(bool(causal)), _ptr(out), _out_code(out.dtype), _ptr(lse),
                                        _ptr(dev_status), _stream_handle(stream))
    _check("attn_fwd_padded", st)
    return out, lse


def attn_fwd_dense_plan(B, Sq, Sk, Hq, Hkv, D, causal=False):
    """(launches, split) attn_fwd_dense makes for these sizes on the current device."""
    n, sp = ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().attn_fwd_dense_plan(B, Sq, Sk, Hq, Hkv, D, int(bool(causal)), ctypes.byref(n),
                                            ctypes.byref(sp))
    _check("attn_fwd_dense_plan", st)
    return n.value, sp.value


def attn_set_wait_give_up(on) -> bool:
    """Make the prefill kernels launched from now on give up their pipeline
    waits at once (a test of the failure path: GBATTN_DEV_TIMEOUT is set,
    the call returns, outputs are undefined); returns the previous setting."""
    prev = ctypes.c_int(0)
    _check("attn_set_wait_give_up", load_library().attn_set_wait_give_up(int(bool(on)), ctypes.byref(prev)))
    return bool(prev.value)


def attn_fwd_varlen_plan(lens_q, D, causal=False, Hq=32, Hkv=8, lens_k=None):
    """Kernel launches attn_fwd_varlen makes for documents of these lengths
    on the current device (host sizes only)."""
    lens_k = lens_q if lens_k is None else lens_k
    n = ctypes.c_int(0)
    st = load_library().attn_fwd_varlen_plan(len(lens_q), int(sum(lens_q)), int(max(list(lens_q) + [0])),
                                             int(max(list(lens_k) + [0])), Hq, Hkv, D, int(bool(causal)),
                                             ctypes.byref(n))
    _check("attn_fwd_varlen_plan", st)
    return n.value


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, softmax_scale=None,
                    causal=False, out=None, lse=None, out_dtype=torch.float32, dev_status=None, stream=None):
    """Packed documents.  q [Tq, Hq, D], k/v [Tk, Hkv, D], cu_seqlens int32
    CUDA tensors [N+1]; max_seqlen_q/k are host ints.  Returns (out [Tq, Hq, D],
    lse [Hq, Tq] or None)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    for n, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    if k.shape != v.shape or k.shape[2] != D:
        raise ValueError("k and v must be [Tk, Hkv, D] matching q")
    n_docs = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() - 1 != n_docs:
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different document counts")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty(Tq, Hq, D, dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty(Hq, Tq, dtype=torch.float32, device=q.device)
    st = load_library().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), n_docs,
                                        Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, D, scale,
                                        int(bool(causal)), _ptr(out), _out_code(out.dtype), _ptr(lse),
                                        _ptr(dev_status), _stream_handle(stream))
    _check("attn_fwd_varlen", st)
    return out, lse


def attn_fwd_paged_workspace_size(num_seqs, Hq, Hkv, D, max_seq_len) -> int:
    return int(load_library().attn_fwd_paged_workspace_size(num_seqs, Hq, Hkv, D, max_seq_len))


def attn_fwd_paged(q, kv_cache, block_table, seq_lens, max_seq_len, softmax_scale=None, causal=True, out=None,
                   lse=None, out_dtype=torch.float32, workspace=None, dev_status=None, stream=None):
    """Decode over a paged cache.  q [S, Hq, D]; kv_cache [2, nb, 128, Hkv, D];
    block_table int32 [S, max_blocks]; seq_lens int32 [S]; max_seq_len host int.
    Returns (out [S, Hq, D], lse [S, Hq] or None).  A workspace tensor of at
    least ``attn_fwd_paged_workspace_size`` bytes may be passed (it is
    allocated here otherwise)."""
    _bf16_cuda("q", q)
    _bf16_cuda("kv_cache", kv_cache)
    S, Hq, D = q.shape
    two, nb, bs, Hkv, Dk = kv_cache.shape
    if two != 2 or Dk != D:
        raise ValueError("kv_cache must be [2, num_blocks, block_size, Hkv, D]")
    for n, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    need = attn_fwd_paged_workspace_size(S, Hq, Hkv, D, int(max_seq_len))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(S, Hq, D, dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty(S, Hq, dtype=torch.float32, device=q.device)
    st = load_library().attn_fwd_paged(_ptr(q), _ptr(kv_cache), nb, bs, _ptr(block_table), block_table.shape[1],
                                       _ptr(seq_lens), S, int(max_seq_len), Hq, Hkv, D, scale, int(bool(causal)),
                                       _ptr(out), _out_code(out.dtype), _ptr(lse), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                       _stream_handle(stream))
    _check("attn_fwd_paged", st)
    return out, lse


def attn_fwd_paged_noalloc(q, kv_cache, block_table, seq_lens, max_seq_len, softmax_scale=None, causal=True,
                           out=None, lse=None, out_dtype=torch.float32, dev_status=None, stream=None):
    """attn_fwd_paged without a workspace argument, for callers that must not
    allocate device memory while it runs (e.g. during CUDA-graph capture): the
    split-K scratch is the library's built-in 32 MiB device array.  Pass
    preallocated ``out`` (and ``lse``) to allocate nothing here either.  The
    first call on a device should happen before any stream capture.  Calls
    that overlap on the GPU share the scratch and race."""
    _bf16_cuda("q", q)
    _bf16_cuda("kv_cache", kv_cache)
    S, Hq, D = q.shape
    two, nb, bs, Hkv, Dk = kv_cache.shape
    if two != 2 or Dk != D:
        raise ValueError("kv_cache must be [2, num_blocks, block_size, Hkv, D]")
    for n, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty(S, Hq, D, dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty(S, Hq, dtype=torch.float32, device=q.device)
    st = load_library().attn_fwd_paged_noalloc(_ptr(q), _ptr(kv_cache), nb, bs, _ptr(block_table),
                                               block_table.shape[1], _ptr(seq_lens), S, int(max_seq_len), Hq, Hkv, D,
                                               scale, int(bool(causal)), _ptr(out), _out_code(out.dtype), _ptr(lse),
                                               _ptr(dev_status), _stream_handle(stream))
    _check("attn_fwd_paged_noalloc", st)
    return out, lse


def attn_kv_cache_write(key, value, slot_mapping, kv_cache, dev_status=None, stream=None):
    """Store key / value [T, Hkv, D] (bf16) into kv_cache [2, nb, bs, Hkv, D]
    in place at slot_mapping [T] (int32 CUDA): token t goes to block
    slot // bs, offset slot % bs; negative slots store nothing."""
    for n, t in (("key", key), ("value", value), ("kv_cache", kv_cache)):
        _bf16_cuda(n, t)
    T, Hkv, D = key.shape
    two, nb, bs, Hc, Dc = kv_cache.shape
    if value.shape != key.shape or two != 2 or (Hc, Dc) != (Hkv, D):
        raise ValueError("key/value must be [T, Hkv, D] and kv_cache [2, num_blocks, block_size, Hkv, D]")
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous() or \
            slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be a contiguous int32 CUDA tensor of T entries")
    st = load_library().attn_kv_cache_write(_ptr(key), _ptr(value), _ptr(slot_mapping), T, _ptr(kv_cache), nb, bs,
                                            Hkv, D, _ptr(dev_status), _stream_handle(stream))
    _check("attn_kv_cache_write", st)
    return kv_cache


def attn_fwd_paged_prefill(q, kv_cache, block_table, seq_lens, cu_seqlens_q, max_seqlen_q, max_seq_len,
                           softmax_scale=None, causal=True, out=None, lse=None, out_dtype=torch.float32,
                           dev_status=None, stream=None):
    """Several query tokens per sequence (packed by cu_seqlens_q, the last
    tokens of each context) against the paged cache.  Returns
    (out [Tq, Hq, D], lse [Hq, Tq] or None); max_seqlen_q / max_seq_len are
    host ints."""
    _bf16_cuda("q", q)
    _bf16_cuda("kv_cache", kv_cache)
    Tq, Hq, D = q.shape
    two, nb, bs, Hkv, Dk = kv_cache.shape
    if two != 2 or Dk != D:
        raise ValueError("kv_cache must be [2, num_blocks, block_size, Hkv, D]")
    for n, t in (("block_table", block_table), ("seq_lens", seq_lens), ("cu_seqlens_q", cu_seqlens_q)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty(Tq, Hq, D, dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty(Hq, Tq, dtype=torch.float32, device=q.device)
    S = cu_seqlens_q.numel() - 1
    st = load_library().attn_fwd_paged_prefill(_ptr(q), _ptr(kv_cache), nb, bs, _ptr(block_table),
                                               block_table.shape[1], _ptr(seq_lens), _ptr(cu_seqlens_q), S, Tq,
                                               int(max_seqlen_q), int(max_seq_len), Hq, Hkv, D, scale,
                                               int(bool(causal)), _ptr(out), _out_code(out.dtype), _ptr(lse),
                                               _ptr(dev_status), _stream_handle(stream))
    _check("attn_fwd_paged_prefill", st)
    return out, lse


def attn_mask_to_varlen(mask, stream=None):
    """mask [B, S] (bool or uint8 CUDA, nonzero = token) -> (cu_seqlens [B+1], packed_pos [B*S]) int32."""
    if mask.dim() != 2 or not mask.is_cuda or mask.element_size() != 1:
        raise ValueError("mask must be a [B, S] bool / uint8 CUDA tensor")
    mask = mask.contiguous()
    B, S = mask.shape
    cu = torch.empty(B + 1, dtype=torch.int32, device=mask.device)
    pos = torch.empty(B * S, dtype=torch.int32, device=mask.device)
    st = load_library().attn_mask_to_varlen(_ptr(mask), B, S, _ptr(cu), _ptr(pos), _stream_handle(stream))
    _check("attn_mask_to_varlen", st)
    return cu, pos


def attn_pack_rows(x, packed_pos, cu_seqlens, stream=None):
    """x [B, S, ...] contiguous CUDA -> packed [B*S, ...]: the masked-in rows in order, then zero rows."""
    B, S = x.shape[:2]
    packed = torch.empty((B * S,) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    rb = x[0, 0].numel() * x.element_size()
    st = load_library().attn_pack_rows(_ptr(x), _ptr(packed_pos), _ptr(cu_seqlens), B, S, rb, _ptr(packed),
                                       _stream_handle(stream))
    _check("attn_pack_rows", st)
    return packed


def attn_unpack_rows(packed, packed_pos, B, S, stream=None):
    """packed [B*S, ...] -> [B, S, ...] with zeros at the padding."""
    out = torch.empty((B, S) + tuple(packed.shape[1:]), dtype=packed.dtype, device=packed.device)
    rb = packed[0].numel() * packed.element_size()
    st = load_library().attn_unpack_rows(_ptr(packed), _ptr(packed_pos), B, S, rb, _ptr(out), _stream_handle(stream))
    _check("attn_unpack_rows", st)
    return out


def attn_unpack_lse(lse_packed, packed_pos, B, S, stream=None):
    """lse_packed [H, B*S] -> [B, H, S], -inf at the padding."""
    H = lse_packed.shape[0]
    lse = torch.empty(B, H, S, dtype=torch.float32, device=lse_packed.device)
    st = load_library().attn_unpack_lse(_ptr(lse_packed), _ptr(packed_pos), B, H, S, _ptr(lse), _stream_handle(stream))
    _check("attn_unpack_lse", st)
    return lse


def attn_fwd_masked(q, k, v, mask, softmax_scale=None, causal=False, cross=False, lse=False, out_dtype=torch.float32,
                    dev_status=None, stream=None):
    """Padded batch q [B, Sq, Hq, D], k/v [B, Sk, Hkv, D] with a [B, Sk]
    padding mask: the masked-in tokens are packed, attended as varlen
    documents and put back (zeros, lse -inf at the padding).  cross=True:
    the mask covers the keys only and every query row is kept.  Returns
    (out [B, Sq, Hq, D], lse [B, Hq, Sq] or None)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    if not cross and Sq != Sk:
        raise ValueError("self-attention needs Sq == Sk (use cross=True for a key-only mask)")
    cu_k, pos_k = attn_mask_to_varlen(mask, stream)
    kp, vp = attn_pack_rows(k, pos_k, cu_k, stream), attn_pack_rows(v, pos_k, cu_k, stream)
    if cross:
        qp = q.view(B * Sq, Hq, D)
        cu_q = torch.arange(0, (B + 1) * Sq, Sq, dtype=torch.int32, device=q.device)
    else:
        qp, cu_q = attn_pack_rows(q, pos_k, cu_k, stream), cu_k
    out_p, lse_p = attn_fwd_varlen(qp, kp, vp, cu_q, cu_k, Sq, Sk, softmax_scale, causal, lse=True if lse else None,
                                   out_dtype=out_dtype, dev_status=dev_status, stream=stream)
    if cross:
        out = out_p.view(B, Sq, Hq, D)
        lse_out = lse_p.view(Hq, B, Sq).permute(1, 0, 2) if lse else None
    else:
        out = attn_unpack_rows(out_p, pos_k, B, Sq, stream)
        lse_out = attn_unpack_lse(lse_p, pos_k, B, Sq, stream) if lse else None
    return out, lse_out


def attn_vsa_layout(prefix_segments, video_shape, tile=(4, 4, 4), block=64):
    """Token blocks of block-sparse video attention (host computation).
    Returns (order int32 [tokens], block_start int32 [NB + 1], n_prefix_blocks)."""
    lib = load_library()
    seg = (ctypes.c_int32 * max(1, len(prefix_segments)))(*[int(x) for x in prefix_segments])
    nb, npre = ctypes.c_int(0), ctypes.c_int(0)
    t, h, w = (int(x) for x in video_shape)
    args = (seg, len(prefix_segments), t, h, w, int(tile[0]), int(tile[1]), int(tile[2]), int(block))
    _check("attn_vsa_layout", lib.attn_vsa_layout(*args, None, None, ctypes.byref(nb), ctypes.byref(npre)))
    order = torch.empty(sum(int(x) for x in prefix_segments) + t * h * w, dtype=torch.int32)
    start = torch.empty(nb.value + 1, dtype=torch.int32)
    _check("attn_vsa_layout", lib.attn_vsa_layout(*args, _ptr(order), _ptr(start), ctypes.byref(nb),
                                                  ctypes.byref(npre)))
    return order, start, npre.value


def attn_vsa_tile_map(prefix_segments, video_shape, tile=(4, 4, 4)):
    """Tiled layout of block-sparse video attention (host computation, 64-token
    blocks).  Returns (tile_index int32 [nbp * 64], block_sizes int32 [nb],
    n_prefix_blocks), host tensors."""
    lib = load_library()
    seg = (ctypes.c_int32 * max(1, len(prefix_segments)))(*[int(x) for x in prefix_segments])
    nb, npre = ctypes.c_int(0), ctypes.c_int(0)
    t, h, w = (int(x) for x in video_shape)
    args = (seg, len(prefix_segments), t, h, w, int(tile[0]), int(tile[1]), int(tile[2]))
    _check("attn_vsa_tile_map", lib.attn_vsa_tile_map(*args, None, None, ctypes.byref(nb), ctypes.byref(npre)))
    index = torch.empty((nb.value + nb.value % 2) * 64, dtype=torch.int32)
    sizes = torch.empty(nb.value, dtype=torch.int32)
    _check("attn_vsa_tile_map", lib.attn_vsa_tile_map(*args, _ptr(index), _ptr(sizes), ctypes.byref(nb),
                                                      ctypes.byref(npre)))
    return index, sizes, npre.value


def attn_gather_rows(src, index, dev_status=None, stream=None):
    """src [N, ...] contiguous CUDA, index int32 CUDA [M] -> dst [M, ...]:
    dst[w] = src[index[w]], zero rows where index[w] < 0."""
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    if index.dtype != torch.int32 or not index.is_cuda or not index.is_contiguous():
        raise ValueError("index must be a contiguous int32 CUDA tensor")
    M = index.numel()
    dst = torch.empty((M,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    rb = src[0].numel() * src.element_size() if src.shape[0] > 0 else dst[0].numel() * dst.element_size()
    st = load_library().attn_gather_rows(_ptr(src), src.shape[0], _ptr(index), M, rb, _ptr(dst), _ptr(dev_status),
                                         _stream_handle(stream))
    _check("attn_gather_rows", st)
    return dst


def attn_vsa_pool(x_tiled, block_sizes, dev_status=None, stream=None):
    """x_tiled [rows >= nb * 64, H, D] bf16 CUDA, block_sizes int32 CUDA [nb]
    -> pooled [H, nb, D] fp32 block means."""
    _bf16_cuda("x_tiled", x_tiled)
    if block_sizes.dtype != torch.int32 or not block_sizes.is_cuda or not block_sizes.is_contiguous():
        raise ValueError("block_sizes must be a contiguous int32 CUDA tensor")
    nb = block_sizes.numel()
    _, H, D = x_tiled.shape
    if x_tiled.shape[0] < nb * 64:
        raise ValueError("x_tiled has fewer than 64 rows per block")
    pooled = torch.empty(H, nb, D, dtype=torch.float32, device=x_tiled.device)
    st = load_library().attn_vsa_pool(_ptr(x_tiled), nb, H, D, _ptr(block_sizes), _ptr(pooled), _ptr(dev_status),
                                      _stream_handle(stream))
    _check("attn_vsa_pool", st)
    return pooled


def attn_vsa_list_size(num_blocks, num_prefix_blocks, topk, Hq) -> int:
    n = ctypes.c_longlong(0)
    _check("attn_vsa_list_size", load_library().attn_vsa_list_size(num_blocks, num_prefix_blocks, topk, Hq,
                                                                   ctypes.byref(n)))
    return n.value


def attn_vsa_block_map(pooled_q, pooled_k, block_sizes, num_prefix_blocks, topk, softmax_scale, dev_status=None,
                       stream=None):
    """pooled_q [Hq, nb, D], pooled_k [Hkv, nb, D] fp32 CUDA -> (kv_list, kv_num)
    int32: per head and tile (query blocks 2t, 2t+1), the union of the key
    blocks they keep, entries (block << 9) | (size << 2) | bits."""
    if pooled_q.dim() != 3 or pooled_k.dim() != 3 or pooled_q.shape[1:] != pooled_k.shape[1:]:
        raise ValueError("pooled_q must be [Hq, nb, D] and pooled_k [Hkv, nb, D] with the same nb and D")
    if pooled_q.dtype != torch.float32 or pooled_k.dtype != torch.float32:
        raise ValueError("pooled_q and pooled_k must be float32")
    Hq, nb, D = pooled_q.shape
    Hkv = pooled_k.shape[0]
    if block_sizes.numel() != nb or block_sizes.dtype != torch.int32:
        raise ValueError(f"block_sizes must hold {nb} int32 entries (one per block)")
    for n_, t in (("pooled_q", pooled_q), ("pooled_k", pooled_k), ("block_sizes", block_sizes)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n_} must be a contiguous CUDA tensor")
    n = attn_vsa_list_size(nb, num_prefix_blocks, topk, Hq)
    kv_list = torch.empty(max(n, 1), dtype=torch.int32, device=pooled_q.device)
    kv_num = torch.empty(Hq, (nb + 1) // 2, dtype=torch.int32, device=pooled_q.device)
    st = load_library().attn_vsa_block_map(_ptr(pooled_q), _ptr(pooled_k), nb, num_prefix_blocks, Hq, Hkv, D, topk,
                                           float(softmax_scale), _ptr(block_sizes), _ptr(kv_list), _ptr(kv_num),
                                           _ptr(dev_status), _stream_handle(stream))
    _check("attn_vsa_block_map", st)
    return kv_list, kv_num


def _check_vsa_fwd_shapes(q_tiled, k_tiled, v_tiled, kv_list, kv_num, num_blocks, num_prefix_blocks, topk,
                          out_index, out_rows, out, lse):
    """Raise ValueError unless the tensors have the sizes the C call derives
    from (num_blocks, Hq, Hkv, D): its tensor maps and list reads trust them."""
    if q_tiled.dim() != 3 or k_tiled.dim() != 3 or v_tiled.dim() != 3:
        raise ValueError("q_tiled, k_tiled and v_tiled must be [rows, heads, D]")
    rows, Hq, D = q_tiled.shape
    want = (num_blocks + num_blocks % 2) * 64
    if rows != want:
        raise ValueError(f"q_tiled has {rows} rows; {num_blocks} blocks need {want} (64 per block, even count)")
    if k_tiled.shape != v_tiled.shape or k_tiled.shape[0] != rows or k_tiled.shape[2] != D:
        raise ValueError("k_tiled and v_tiled must both be [rows of q_tiled, Hkv, D of q_tiled]")
    for n_, t in (("kv_list", kv_list), ("kv_num", kv_num)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{n_} must be a contiguous int32 tensor")
    need = attn_vsa_list_size(num_blocks, num_prefix_blocks, topk, Hq)
    if kv_list.numel() < need:
        raise ValueError(f"kv_list holds {kv_list.numel()} entries; these sizes need {need}")
    if tuple(kv_num.shape) != (Hq, (num_blocks + 1) // 2):
        raise ValueError(f"kv_num must be [Hq, (num_blocks + 1) // 2] = [{Hq}, {(num_blocks + 1) // 2}]")
    if out_index is not None and (out_index.dtype != torch.int32 or out_index.numel() != rows):
        raise ValueError(f"out_index must hold {rows} int32 entries (one per tiled row)")
    if out_index is None and out_rows != rows:
        raise ValueError("without out_index the output stays tiled: out_rows must equal the tiled row count")
    if out is not None and tuple(out.shape) != (out_rows, Hq, D):
        raise ValueError(f"out must be [out_rows, Hq, D] = [{out_rows}, {Hq}, {D}]")
    if torch.is_tensor(lse) and (tuple(lse.shape) != (Hq, out_rows) or lse.dtype != torch.float32):
        raise ValueError(f"lse must be float32 [Hq, out_rows] = [{Hq}, {out_rows}]")


def attn_fwd_vsa(q_tiled, k_tiled, v_tiled, kv_list, kv_num, num_blocks, num_prefix_blocks, topk, out_index=None,
                 out_rows=None, softmax_scale=None, lse=None, out_dtype=torch.float32, out=None, dev_status=None,
                 stream=None):
    """Block-sparse attention over tiled q [nbp*64, Hq, D], k/v [nbp*64, Hkv, D]
    (bf16 CUDA) and the lists of attn_vsa_block_map.  Row r of the tiled layout
    goes to out row out_index[r] (None: out stays tiled).  Returns (out
    [out_rows, Hq, D], lse [Hq, out_rows] or None)."""
    if out_rows is None:
        out_rows = q_tiled.shape[0]
    _check_vsa_fwd_shapes(q_tiled, k_tiled, v_tiled, kv_list, kv_num, num_blocks, num_prefix_blocks, topk,
                          out_index, out_rows, out, lse)
    for n_, t in (("q_tiled", q_tiled), ("k_tiled", k_tiled), ("v_tiled", v_tiled)):
        _bf16_cuda(n_, t)
    for n_, t in (("kv_list", kv_list), ("kv_num", kv_num), ("out_index", out_index), ("out", out), ("lse", lse)):
        if torch.is_tensor(t) and not t.is_cuda:
            raise ValueError(f"{n_} must be a CUDA tensor")
    rows, Hq, D = q_tiled.shape
    Hkv = k_tiled.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(out_rows, Hq, D, dtype=out_dtype, device=q_tiled.device)
    if lse is True:
        lse = torch.empty(Hq, out_rows, dtype=torch.float32, device=q_tiled.device)
    st = load_library().attn_fwd_vsa(_ptr(q_tiled), _ptr(k_tiled), _ptr(v_tiled), num_blocks, num_prefix_blocks, topk,
                                     _ptr(kv_list), _ptr(kv_num), _ptr(out_index), out_rows, Hq, Hkv, D,
                                     float(softmax_scale), _ptr(out), _out_code(out.dtype), _ptr(lse),
                                     _ptr(dev_status), _stream_handle(stream))
    _check("attn_fwd_vsa", st)
    return out, lse


class VsaPlan:
    """One geometry's tiled layout, computed on the host once and kept on the
    device (the page caches the same metadata per geometry)."""

    def __init__(self, prefix_segments, video_shape, device, tile=(4, 4, 4)):
        index, sizes, npre = attn_vsa_tile_map(prefix_segments, video_shape, tile)
        self.tokens = sum(int(x) for x in prefix_segments) + math.prod(int(x) for x in video_shape)
        self.num_blocks = sizes.numel()
        self.num_prefix_blocks = npre
        self.rows = index.numel()
        self.tile_index = index.to(device)
        self.block_sizes = sizes.to(device)


def attn_vsa(q, k, v, plan: VsaPlan, topk=64, softmax_scale=None, lse=False, out_dtype=torch.float32,
             dev_status=None, stream=None):
    """Block-sparse video attention of one sequence: q [S, Hq, D], k/v [S, Hkv, D]
    bf16 CUDA, S = plan.tokens.  Tiles q, k, v, pools q and k, builds the block
    map and attends it; returns (out [S, Hq, D], lse [Hq, S] or None)."""
    for n_, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n_, t)
    S, Hq, D = q.shape
    if S != plan.tokens or k.shape[0] != S or v.shape[0] != S:
        raise ValueError(f"the plan's geometry has {plan.tokens} tokens, q/k/v have {S}")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    qt = attn_gather_rows(q, plan.tile_index, dev_status, stream)
    kt = attn_gather_rows(k, plan.tile_index, dev_status, stream)
    vt = attn_gather_rows(v, plan.tile_index, dev_status, stream)
    pq = attn_vsa_pool(qt, plan.block_sizes, dev_status, stream)
    pk = attn_vsa_pool(kt, plan.block_sizes, dev_status, stream)
    kv_list, kv_num = attn_vsa_block_map(pq, pk, plan.block_sizes, plan.num_prefix_blocks, topk, softmax_scale,
                                         dev_status, stream)
    return attn_fwd_vsa(qt, kt, vt, kv_list, kv_num, plan.num_blocks, plan.num_prefix_blocks, topk,
                        out_index=plan.tile_index, out_rows=S, softmax_scale=softmax_scale,
                        lse=True if lse else None, out_dtype=out_dtype, dev_status=dev_status, stream=stream)
