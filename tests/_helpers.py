"""Shared helpers for the GPU parity tests (no attention arithmetic here)."""

import numpy as np
import torch

OUT_TOL = 1e-2   # max |out - oracle|, fp32 output
LSE_TOL = 1e-3   # max |lse - oracle|


def dev():
    return torch.device("cuda:0")


def status_word():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def to_np(t):
    return t.detach().cpu().double().numpy()


def max_err(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb), "finite / non-finite pattern differs"
    assert np.array_equal(a[~fa], b[~fb]), "non-finite values differ"
    return float(np.max(np.abs(a[fa] - b[fb]))) if fa.any() else 0.0


def assert_close(out, lse, ref_out, ref_lse, out_tol=OUT_TOL, lse_tol=LSE_TOL, what=""):
    eo = max_err(to_np(out) if torch.is_tensor(out) else out, ref_out)
    assert eo <= out_tol, f"{what}: max |out err| {eo:.3e} > {out_tol}"
    if lse is not None:
        el = max_err(to_np(lse) if torch.is_tensor(lse) else lse, ref_lse)
        assert el <= lse_tol, f"{what}: max |lse err| {el:.3e} > {lse_tol}"


def bf16_half_ulp(x):
    """Half a bf16 ulp of |x| (the rounding bound of a bf16 output)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


# ---- block-sparse video attention: the per-tile list format of attn_vsa_block_map
def _list_size(nb, npre, topk, hq):
    import attention_forward_09_gb300 as gb
    return gb.attn_vsa_list_size(nb, npre, topk, hq)


def vsa_tile_offsets(nb, npre, topk):
    """Start and capacity of each tile's list within one head (the placement
    rule stated with attn_vsa_block_map)."""
    nt, keep = (nb + 1) // 2, min(topk, nb - npre)
    td = nt if keep == nb - npre else min(nt, (npre + 1) // 2)
    c2 = min(nb, npre + 2 * keep)
    return [(t * nb, nb) if t < td else (td * nb + (t - td) * c2, c2) for t in range(nt)]


def vsa_lists_from_map(bm, sizes, npre, topk):
    """Host encoding of a bool block map [Hq, nb, nb] into the kernel's lists
    (CPU tensors)."""
    hq, nb, _ = bm.shape
    per_head = _list_size(nb, npre, topk, 1)
    kl = np.zeros(max(hq * per_head, 1), dtype=np.int32)
    kn = np.zeros((hq, (nb + 1) // 2), dtype=np.int32)
    for h in range(hq):
        for t, (off, cap) in enumerate(vsa_tile_offsets(nb, npre, topk)):
            r1 = bm[h, 2 * t + 1] if 2 * t + 1 < nb else np.zeros(nb, bool)
            bits = bm[h, 2 * t].astype(int) | (r1.astype(int) << 1)
            ent = [(j << 9) | (int(sizes[j]) << 2) | want for want in (3, 1, 2) for j in range(nb) if bits[j] == want]
            assert len(ent) <= cap
            kl[h * per_head + off:h * per_head + off + len(ent)] = ent
            kn[h, t] = len(ent)
    return torch.from_numpy(kl), torch.from_numpy(kn)


def vsa_map_from_lists(kv_list, kv_num, nb, npre, topk, sizes):
    """The kernel's lists -> bool map [Hq, nb, nb], checking their format."""
    kl, kn = kv_list.cpu().numpy(), kv_num.cpu().numpy()
    hq = kn.shape[0]
    per_head = _list_size(nb, npre, topk, 1)
    bm = np.zeros((hq, nb, nb), dtype=bool)
    for h in range(hq):
        for t, (off, cap) in enumerate(vsa_tile_offsets(nb, npre, topk)):
            n = int(kn[h, t])
            assert 0 <= n <= cap
            e = kl[h * per_head + off:h * per_head + off + n].astype(np.int64)
            blk, sz, bits = e >> 9, (e >> 2) & 127, e & 3
            assert np.all(bits != 0) and np.array_equal(sz, np.asarray(sizes)[blk])
            rank = np.array([0, 1, 2, 0])[bits]  # groups: kept by both, by the first only, by the second only
            assert np.all(np.diff(rank) >= 0) and np.all(np.diff(blk)[np.diff(rank) == 0] > 0)
            bm[h, 2 * t, blk[(bits & 1) != 0]] = True
            if 2 * t + 1 < nb:
                bm[h, 2 * t + 1, blk[(bits & 2) != 0]] = True
            else:
                assert not np.any(bits & 2)
    return bm
