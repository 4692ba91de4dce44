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


def tag_values(j, hkv):
    """The four tag dims of key j (int or array) in kv head hkv: every value is
    an integer in [1, 256], exact in bf16 and never 0 (so a tiny weight on
    another key can never survive rounding in place of an exact 0)."""
    return ((j % 256) + 1, (j // 256) + 1, hkv + 1, ((5 * j + 3) % 256) + 1)


def position_tags(sk, hk, d):
    """V rows that spell out their own key index j and kv head exactly in bf16
    (dims 0..3 = tag_values(j, kv head)); the remaining dims are 0."""
    v = torch.zeros(sk, hk, d, dtype=torch.float32)
    j = torch.arange(sk, dtype=torch.int64)
    for h in range(hk):
        t = tag_values(j, h)
        for k in range(4):
            v[:, h, k] = t[k].float() if torch.is_tensor(t[k]) else float(t[k])
    return v


def decode_tag(row):
    """Inverse of ``position_tags`` for one output row: (j, kv_head)."""
    lo = int(round(float(row[0]))) - 1
    hi = int(round(float(row[1]))) - 1
    return lo + 256 * hi, int(round(float(row[2]))) - 1


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
