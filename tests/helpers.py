"""Test-side helpers: place logical per-sequence K/V rows into a paged cache and
compare results.  Input construction only; no attention arithmetic."""
import numpy as np
import torch


def scatter_logical(w, k_logical, v_logical):
    """Write per-sequence logical rows into ``w``'s paged caches.

    ``k_logical[s]`` / ``v_logical[s]``: float tensors [S_k(s), H_k, d]; they are
    rounded to bf16 and stored at block_table[s][j // b], slot j % b.
    """
    bt = w.block_table.cpu()
    for s in range(w.num_seqs):
        sk = w.seqlens_k[s]
        for j0 in range(0, sk, w.b):
            blk = int(bt[s, j0 // w.b])
            n = min(w.b, sk - j0)
            w.k_cache[blk, :n] = k_logical[s][j0:j0 + n].to(torch.bfloat16).to(w.k_cache.device)
            w.v_cache[blk, :n] = v_logical[s][j0:j0 + n].to(torch.bfloat16).to(w.v_cache.device)


def gather_logical(w, cache, s):
    """The logical rows [S_k(s), H_k, d] of sequence s, read back through the table."""
    bt = w.block_table.cpu()
    sk = w.seqlens_k[s]
    rows = []
    for j0 in range(0, sk, w.b):
        blk = int(bt[s, j0 // w.b])
        rows.append(cache[blk, :min(w.b, sk - j0)].cpu())
    if not rows:
        return torch.zeros(0, w.hk, w.d, dtype=cache.dtype)
    return torch.cat(rows, 0)


def position_tags(sk, hk, d):
    """V rows that spell out their own key index j and kv head exactly in bf16:
    dim 0 = j mod 256, dim 1 = j // 256, dim 2 = kv head, dim 3 = (5 j + 3) mod 256,
    the remaining dims 0."""
    v = torch.zeros(sk, hk, d, dtype=torch.float32)
    j = torch.arange(sk, dtype=torch.float32)
    for h in range(hk):
        v[:, h, 0] = torch.remainder(j, 256)
        v[:, h, 1] = torch.div(j, 256, rounding_mode="floor")
        v[:, h, 2] = h
        v[:, h, 3] = torch.remainder(5 * j + 3, 256)
    return v


def decode_tag(row):
    """Inverse of ``position_tags`` for one output row: (j, kv_head)."""
    return int(round(float(row[0]) + 256 * float(row[1]))), int(round(float(row[2])))


def token_of_row(w):
    """(seq, local index i, ctx) for every packed token."""
    out = []
    for s, (sq, sk) in enumerate(zip(w.seqlens_q, w.seqlens_k)):
        for i in range(sq):
            out.append((s, i, sk - sq))
    return out


def max_mean_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    diff = np.abs(a - b)
    if diff.size == 0:
        return 0.0, 0.0
    return float(diff.max()), float(diff.mean())
