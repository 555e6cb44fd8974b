"""Float64 CPU oracle for the fused scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA path.

What it computes (the plain definition, score matrix materialised):

    s[i, j]  = scale * <q[i, h], k[j, kv(h)]>           for visible (i, j)
    out[i,h] = sum_j exp(s[i,j] - M_i) v[j, kv(h)] / sum_j exp(s[i,j] - M_i)
    lse[h,i] = M_i + ln sum_j exp(s[i,j] - M_i),        M_i = max_j s[i,j]

Sources, by page and section:

* Output and log-sum-exp pair: vllm-omni ``flash_attn.py``,
  ``FlashAttentionImpl._unwrap_flash_output`` (the FlashAttention call may
  return ``(out, lse)``); vllm-ascend ``attention_v1.py``,
  ``AscendAttentionBackendImpl.full_graph_fia`` (``softmax_lse`` output).
* Explicit softmax scale: ``flash_attn.py``, ``FlashAttentionImpl.__init__``.
* Causal masking is bottom-right aligned: ``flash_attn.py``,
  ``FlashAttentionImpl.forward_fa_npu`` -- key position kp is blocked for query
  position qp iff ``kp > qp + (Sk - Sq)``.
* Rows with no visible key ("invalid-row handling" in ``forward_fa_npu``):
  reading taken here -- out = 0 and lse = -inf, which also matches the
  "padded rows come back zero" convention of vllm-omni ``fastvideo_vsa.py``
  (SDPA fallback with packed padding).
* GQA: ``attention_v1.py``, ``AscendAttentionBackendImpl.__init__``
  (``num_heads % num_kv_heads == 0``, ``num_queries_per_kv``); reading taken
  here -- query head h reads KV head ``h // (Hq // Hkv)``.
* Packed documents: ``flash_attn.py``, ``FlashAttentionImpl._forward_varlen_packed``
  (attention only inside ``[cu_seqlens[i], cu_seqlens[i+1])``) and
  ``FlashAttentionImpl._flash_varlen_wrapper`` (dense == varlen with
  ``arange`` cu_seqlens).
* Paged cache ``(2, num_blocks, block_size, num_kv_heads, head_size)``:
  ``attention_v1.py``, ``AscendAttentionBackend.get_kv_cache_shape``; token t
  of sequence s sits at slot ``block_table[s, t // block_size] * block_size +
  t % block_size`` (``AscendMetadata.slot_mapping`` comment);
  ``AscendAttentionBackendImpl.forward_paged_attention`` reads the cache
  through ``block_tables`` and ``seq_lens`` (``context_lens``).

Every array argument is converted to float64 first; bf16 inputs convert
exactly, so the oracle sees the same numbers the kernels see.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """Exact conversion to a float64 ndarray (torch tensors go through float32)."""
    if hasattr(x, "detach"):  # torch tensor; bf16 -> fp32 is exact
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.asarray(x, dtype=np.int64)


def visible_mask(lq: int, lk: int, causal: bool, rows=None) -> np.ndarray:
    """Boolean [len(rows), lk]: True where query row i may attend key j.

    Non-causal: every key of the document.  Causal: bottom-right aligned,
    j <= i + (lk - lq) (``flash_attn.py``, ``FlashAttentionImpl.forward_fa_npu``).
    """
    i = np.arange(lq) if rows is None else np.asarray(rows, dtype=np.int64)
    j = np.arange(lk)
    if not causal:
        return np.ones((i.size, lk), dtype=bool)
    return j[None, :] <= i[:, None] + (lk - lq)


def attention_single(q, k, v, scale: float, causal: bool, rows=None):
    """One document.

    q: [Lq, Hq, D]; k, v: [Lk, Hkv, D] (any float dtype).
    rows: optional iterable of query rows to evaluate (default: all).
    Returns out [R, Hq, D] and lse [Hq, R] (float64), R = number of rows.
    Rows that see no key get out = 0 and lse = -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lq, hq, d = q.shape
    lk, hkv, dk = k.shape
    if dk != d or v.shape != k.shape:
        raise ValueError("k and v must both be [Lk, Hkv, D] with D matching q")
    if hkv == 0 or hq % hkv != 0:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    group = hq // hkv
    rows = np.arange(lq) if rows is None else np.asarray(rows, dtype=np.int64)
    r = rows.size
    out = np.zeros((r, hq, d))
    lse = np.full((hq, r), -np.inf)
    if r == 0 or lk == 0:
        return out, lse
    vis = visible_mask(lq, lk, causal, rows)
    live = vis.any(axis=1)
    for h in range(hq):
        kv = h // group
        s = scale * (q[rows, h, :] @ k[:, kv, :].T)  # [R, Lk]
        s = np.where(vis, s, -np.inf)
        m = np.where(live, s.max(axis=1), 0.0)
        p = np.where(vis, np.exp(s - m[:, None]), 0.0)
        l = p.sum(axis=1)
        num = p @ v[:, kv, :]
        out[live, h, :] = num[live] / l[live, None]
        lse[h, live] = m[live] + np.log(l[live])
    return out, lse


def attention_dense(q, k, v, scale: float, causal: bool):
    """Fixed-length batch (vllm-omni ``flash_attn.py``, dense ``flash_attn_func`` route).

    q: [B, Sq, Hq, D]; k, v: [B, Sk, Hkv, D].
    Returns out [B, Sq, Hq, D] and lse [B, Hq, Sq].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, sq, hq, d = q.shape
    out = np.zeros((b, sq, hq, d))
    lse = np.full((b, hq, sq), -np.inf)
    for bi in range(b):
        out[bi], lse[bi] = attention_single(q[bi], k[bi], v[bi], scale, causal)
    return out, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool):
    """Packed documents (``flash_attn.py``, ``FlashAttentionImpl._forward_varlen_packed``).

    q: [Tq, Hq, D]; k, v: [Tk, Hkv, D]; cu_seqlens_q/k: [N+1] non-decreasing,
    starting at 0 and ending at Tq / Tk.  Document n owns query rows
    [cu_q[n], cu_q[n+1]) and key rows [cu_k[n], cu_k[n+1]); nothing attends
    across documents.  Returns out [Tq, Hq, D] and lse [Hq, Tq].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck = _i64(cu_seqlens_q), _i64(cu_seqlens_k)
    check_cu_seqlens(cq, q.shape[0])
    check_cu_seqlens(ck, k.shape[0])
    if cq.size != ck.size:
        raise ValueError("cu_seqlens_q and cu_seqlens_k describe different document counts")
    tq, hq, d = q.shape
    out = np.zeros((tq, hq, d))
    lse = np.full((hq, tq), -np.inf)
    for n in range(cq.size - 1):
        qs, qe, ks, ke = cq[n], cq[n + 1], ck[n], ck[n + 1]
        o, l = attention_single(q[qs:qe], k[ks:ke], v[ks:ke], scale, causal)
        out[qs:qe] = o
        lse[:, qs:qe] = l
    return out, lse


def check_cu_seqlens(cu, total: int) -> None:
    cu = _i64(cu)
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) < 0):
        raise ValueError(f"cu_seqlens must start at 0, be non-decreasing and end at {total}")


def paged_gather(kv_cache, block_table, seq_lens):
    """Contiguous K and V of each sequence read through its block table.

    kv_cache: [2, num_blocks, block_size, Hkv, D]; block_table: [S, max_blocks];
    seq_lens: [S].  Token t of sequence s is slot ``block_table[s, t // bs] *
    bs + t % bs`` (``attention_v1.py``, ``AscendMetadata.slot_mapping``).
    Only the gathered rows are converted to float64.
    Returns two lists of [L_s, Hkv, D] float64 arrays.
    """
    bt, sl = _i64(block_table), _i64(seq_lens)
    _, nb, bs, hkv, d = kv_cache.shape
    ks, vs = [], []
    for s in range(sl.size):
        t = np.arange(sl[s])
        blocks = bt[s, t // bs]
        if t.size and (blocks.min() < 0 or blocks.max() >= nb):
            raise ValueError(f"block_table row {s} points outside the cache")
        slots = t % bs
        if hasattr(kv_cache, "detach"):  # torch tensor: index first, then convert
            import torch

            bi, si = torch.from_numpy(blocks), torch.from_numpy(slots)
            ks.append(_f64(kv_cache[0][bi, si]))
            vs.append(_f64(kv_cache[1][bi, si]))
        else:
            ks.append(_f64(np.asarray(kv_cache)[0][blocks, slots]))
            vs.append(_f64(np.asarray(kv_cache)[1][blocks, slots]))
    return ks, vs


def kv_cache_write(key, value, slot_mapping, kv_cache):
    """The cache after writing each token's K and V at its slot
    (vllm-ascend ``attention_v1.py``, ``AscendAttentionBackendImpl.reshape_and_cache``;
    the slot rule is the ``AscendMetadata.slot_mapping`` comment: slot
    ``block * block_size + offset``).

    key, value: [T, Hkv, D]; slot_mapping: [T] ints; kv_cache:
    [2, num_blocks, block_size, Hkv, D].  Token t goes to
    ``cache[0 / 1, slot // block_size, slot % block_size]``.  A negative slot
    stores nothing (the padding-token convention); a slot past the cache is an
    error.  Tokens are written in order, so a repeated slot keeps the last
    token.  A pure copy: the result holds the input bits, in the cache's dtype.
    Returns a new tensor / array; the input cache is not modified.
    """
    _, nb, bs, hkv, d = kv_cache.shape
    slots = _i64(slot_mapping)
    if key.shape[0] != slots.size or value.shape[0] != slots.size:
        raise ValueError("key, value and slot_mapping disagree on the token count")
    out = kv_cache.clone() if hasattr(kv_cache, "clone") else np.array(kv_cache, copy=True)
    for t in range(slots.size):
        slot = int(slots[t])
        if slot < 0:
            continue
        if slot >= nb * bs:
            raise ValueError(f"slot {slot} of token {t} is past the cache ({nb} blocks of {bs})")
        block, offset = divmod(slot, bs)
        out[0, block, offset] = key[t]
        out[1, block, offset] = value[t]
    return out


def attention_paged(q, kv_cache, block_table, seq_lens, scale: float):
    """Decode over a paged cache (``attention_v1.py``, ``forward_paged_attention``).

    q: [S, Hq, D], one query token per sequence.  With one query the
    bottom-right causal mask shows it the whole context, so causal has no
    effect here.  Returns out [S, Hq, D] and lse [S, Hq].
    """
    q = _f64(q)
    s_count, hq, d = q.shape
    ks, vs = paged_gather(kv_cache, block_table, seq_lens)
    out = np.zeros((s_count, hq, d))
    lse = np.full((s_count, hq), -np.inf)
    for s in range(s_count):
        o, l = attention_single(q[s:s + 1], ks[s], vs[s], scale, causal=False)
        out[s] = o[0]
        lse[s] = l[:, 0]
    return out, lse


def attention_paged_prefill(q, kv_cache, block_table, seq_lens, cu_seqlens_q, scale: float, causal: bool):
    """Several query tokens per sequence over the paged cache: chunked
    prefill and speculative decode (vllm-ascend ``attention_v1.py``,
    ``AscendAttentionState`` PrefillCacheHit / ChunkedPrefill / SpecDecoding,
    served from the cache through ``block_table``).

    q: [Tq, Hq, D] packed by cu_seqlens_q [S + 1]; the q_len_s queries of
    sequence s are the last q_len_s of its seq_lens[s] context tokens, all
    already in the cache.  Causal is bottom-right: query i sees keys
    j <= i + seq_len - q_len.  Returns out [Tq, Hq, D], lse [Hq, Tq].
    """
    cq, sl = _i64(cu_seqlens_q), _i64(seq_lens)
    check_cu_seqlens(cq, q.shape[0])
    ks, vs = paged_gather(kv_cache, block_table, seq_lens)
    tq, hq, d = q.shape
    out = np.zeros((tq, hq, d))
    lse = np.full((hq, tq), -np.inf)
    for s in range(sl.size):
        a, b = int(cq[s]), int(cq[s + 1])
        if b > a:
            o, l = attention_single(q[a:b], ks[s], vs[s], scale, causal)
            out[a:b] = o
            lse[:, a:b] = l
    return out, lse


def attention_masked(q, k, v, mask, scale: float, causal: bool, cross: bool = False):
    """Padded batch with a [B, S] padding mask (vllm-omni ``flash_attn.py``,
    ``FlashAttentionImpl._forward_varlen_masked``): the masked-in tokens of
    each batch row are packed in order, varlen attention runs on the packed
    documents, and the output goes back to the padded positions, zeros at
    the padding.  ``cross``: the mask covers the keys only and every query
    row is kept (the cross-attention branch there).

    q: [B, Sq, Hq, D]; k, v: [B, Sk, Hkv, D]; mask: [B, Sk] (nonzero = token).
    Returns out [B, Sq, Hq, D] and lse [B, Hq, Sq] (-inf at padded rows).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    m = np.asarray(mask.cpu() if hasattr(mask, "cpu") else mask) != 0
    b, sq, hq, d = q.shape
    out = np.zeros((b, sq, hq, d))
    lse = np.full((b, hq, sq), -np.inf)
    for i in range(b):
        keys = np.nonzero(m[i])[0]  # packed order = position order
        rows = np.arange(sq) if cross else keys
        o, l = attention_single(q[i, rows], k[i, keys], v[i, keys], scale, causal)
        out[i, rows] = o
        lse[i][:, rows] = l
    return out, lse


def vsa_blocks(prefix_segments, video_shape, tile=(4, 4, 4), block=64):
    """Token blocks of block-sparse video attention (vllm-omni
    ``fastvideo_vsa.py``, ``_get_h3_tile_metadata``): each prefix segment
    cut into chunks of ``block`` tokens, then the (T, H, W) video grid, whose
    tokens follow the prefix in T, H, W order, cut into ``tile`` boxes taken
    in T, H, W order (boxes at the grid's far edges are smaller).

    Returns (blocks, n_prefix_blocks): blocks is a list of int arrays of
    token indices, each a block in the order the method lays them out.
    """
    blocks, at = [], 0
    for seg in prefix_segments:
        for c0 in range(0, seg, block):
            blocks.append(np.arange(at + c0, at + min(seg, c0 + block)))
        at += seg
    n_prefix = len(blocks)
    t, h, w = video_shape
    grid = np.arange(t * h * w).reshape(t, h, w) + at
    for i in range(0, t, tile[0]):
        for j in range(0, h, tile[1]):
            for k in range(0, w, tile[2]):
                blocks.append(grid[i:i + tile[0], j:j + tile[1], k:k + tile[2]].flatten())
    return blocks, n_prefix


def vsa_pool(x, blocks):
    """Mean token of every block (``fastvideo_vsa.py``, ``_pool_h3_tiles``:
    the block's sum divided by its true token count).  x: [S, H, D].
    Returns [NB, H, D] float64."""
    x = _f64(x)
    return np.stack([x[b].mean(axis=0) for b in blocks])


def vsa_block_map(q, k, blocks, n_prefix, topk: int, scale: float):
    """Block selection (``fastvideo_vsa.py``, ``_pool_h3_tiles`` and
    ``_build_h3_block_map``): the mean query and key of every block, block
    scores scale * mean_q . mean_k per head, then for each query block the
    ``topk`` best video key blocks (ties to the lower block index), plus
    every prefix key block; prefix query blocks keep every key block.

    q, k: [S, Hq, D] / [S, Hkv, D] (one sequence).  Returns bool [Hq, NB, NB].
    """
    q, k = _f64(q), _f64(k)
    hq, hkv = q.shape[1], k.shape[1]
    g = hq // hkv
    nb = len(blocks)
    mq = vsa_pool(q, blocks)  # [NB, Hq, D]
    mk = vsa_pool(k, blocks)  # [NB, Hkv, D]
    n_video = nb - n_prefix
    keep = min(topk, n_video)
    bm = np.zeros((hq, nb, nb), dtype=bool)
    for h in range(hq):
        sc = scale * (mq[:, h, :] @ mk[:, h // g, :].T)  # [NB, NB]
        for i in range(nb):
            if i < n_prefix or keep == n_video:
                bm[h, i, :] = True
                continue
            order = np.argsort(-sc[i, n_prefix:], kind="stable")[:keep] + n_prefix
            bm[h, i, order] = True
            bm[h, i, :n_prefix] = True
    return bm


def attention_block_sparse(q, k, v, blocks, block_map, scale: float):
    """Each query token attends the tokens of the key blocks its block keeps
    (``fastvideo_vsa.py``, the block-sparse forward behind ``_forward_h3``,
    without the trained gate branch), in token order.

    q: [S, Hq, D]; k, v: [S, Hkv, D]; block_map bool [Hq, NB, NB].
    Returns out [S, Hq, D], lse [Hq, S].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    s_len, hq, d = q.shape
    g = hq // k.shape[1]
    out = np.zeros((s_len, hq, d))
    lse = np.full((hq, s_len), -np.inf)
    for h in range(hq):
        kv = h // g
        for i, rows in enumerate(blocks):
            keys = np.concatenate([blocks[j] for j in np.nonzero(block_map[h, i])[0]])
            sc = scale * (q[rows, h, :] @ k[keys, kv, :].T)
            m = sc.max(axis=1)
            p = np.exp(sc - m[:, None])
            l = p.sum(axis=1)
            out[rows, h, :] = (p @ v[keys, kv, :]) / l[:, None]
            lse[h, rows] = m + np.log(l)
    return out, lse


def softmax_weights(q, k, scale: float, causal: bool, head: int):
    """The attention weights of one head, [Lq, Lk] (for invariant checks)."""
    q, k = _f64(q), _f64(k)
    lq, hq, _ = q.shape
    lk, hkv, _ = k.shape
    kv = head // (hq // hkv)
    vis = visible_mask(lq, lk, causal)
    s = np.where(vis, scale * (q[:, head, :] @ k[:, kv, :].T), -np.inf)
    live = vis.any(axis=1)
    m = np.where(live, s.max(axis=1), 0.0)
    p = np.where(vis, np.exp(s - m[:, None]), 0.0)
    l = p.sum(axis=1)
    return np.where(live[:, None], p / np.where(live, l, 1.0)[:, None], 0.0)
