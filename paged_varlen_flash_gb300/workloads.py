"""Seeded synthetic inputs for unified paged varlen attention.

This module only draws inputs: sequence lengths, block tables, and the bf16
Q / K / V values.  It holds none of the attention arithmetic, so the CUDA path
and the CPU oracle can both be fed from it.

Named workloads (the sizes of the five benchmark configurations):

* ``tiny``            1 sequence, S_q = S_k = 128, H_q/H_k = 4/1, d = 64,
                      tau = 1/8, b = 16, 8 blocks drawn from a 32-block pool, causal.
* ``decode``          64 sequences, S_q = 1, S_k ~ U{512..8192}, 32/8, d = 128,
                      b = 16, blocks drawn without replacement from a 40,000-block
                      pool, causal.
* ``chunked``         16 sequences, prior context ~ U{0..4096}, S_q ~ U{1..512},
                      32/8, d = 128, b = 32, pool 4,096 blocks, causal +
                      sliding window 1024 + softcap 50 + per-head sinks ~ N(0,1).
* ``long_prefill``    1 sequence, S_q = S_k = 8192, 128/8, d = 128, b = 64,
                      identity block table (``long_prefill_shuffled``: the same
                      data behind a shuffled table).
* ``wide_mha_alibi``  8 sequences x 4096, 32/32, d = 256, b = 64, shuffled 512-block
                      pool, values 0.5 * N(0,1), causal, ALiBi slopes 2^(-8h/32),
                      h = 1..32.
* ``decode_fp8``      the ``decode`` lengths and tables with an fp8 e4m3 K/V cache
                      (one scale per tensor, 1/32; codes of N(0,1) / scale).
* ``decode_d64`` / ``decode_d256``  the ``decode`` lengths and tables with
                      head size 64 / 256 (the other decode head sizes).
* ``decode_topk``     sparse top-k decode: 256 sequences, S_q = 1,
                      S_k ~ U{4096..16384}, H_q/H_k = 16/1, d = 128, b = 64,
                      pool 48,000 blocks, causal; each query token attends to
                      its own list of 2048 distinct key positions drawn
                      uniformly from its context (random order).

Lengths and block tables come from a CPU ``torch.Generator`` seeded with
``1000 + config index`` and are therefore identical on every device; the bf16
values are drawn on the device the workload is built for (N(0,1) in fp32, then
rounded to bf16).  Key slots that no sequence uses -- blocks outside every
table and the tail of each sequence's last block -- are filled with NaN when
``poison=True`` so that a kernel reading them shows up as NaN in its output;
block-table padding past a sequence's last block holds -1.

fp8 caches (``kv_fp8=True``) hold e4m3 codes as uint8: the N(0,1) values are
divided by the tensor's scale and rounded to e4m3 by PyTorch's
``float8_e4m3fn`` conversion; their poison is the NaN code 0x7f.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

CONFIG_NAMES = ["tiny", "decode", "chunked", "long_prefill", "wide_mha_alibi"]
_CONFIG_INDEX = {
    "tiny": 0, "decode": 1, "chunked": 2, "long_prefill": 3,
    "long_prefill_shuffled": 3, "wide_mha_alibi": 4, "decode_fp8": 1, "decode_topk": 5,
    "decode_d64": 1, "decode_d256": 1,
}


@dataclass
class Workload:
    name: str
    hq: int
    hk: int
    d: int
    b: int
    num_blocks: int
    seqlens_q: List[int]
    seqlens_k: List[int]
    q: torch.Tensor                   # bf16 [total_q, hq, d]
    k_cache: torch.Tensor             # bf16 [num_blocks, b, hk, d]
    v_cache: torch.Tensor             # bf16 [num_blocks, b, hk, d]
    block_table: torch.Tensor         # int32 [num_seqs, max_blocks_per_seq]
    cu_seqlens_q: torch.Tensor        # int32 [num_seqs + 1]
    seqused_k: torch.Tensor           # int32 [num_seqs]
    scale: float
    causal: bool = True
    softcap: float = 0.0              # 0 = off
    window: int = 0                   # 0 = off
    sinks: Optional[torch.Tensor] = None         # fp32 [hq]
    alibi_slopes: Optional[torch.Tensor] = None  # fp32 [hq]
    meta: dict = field(default_factory=dict)
    kv_fp8: bool = False              # caches hold e4m3 codes (uint8)
    k_scale: float = 1.0              # K = e4m3(k) * k_scale when kv_fp8
    v_scale: float = 1.0
    qq_bias: Optional[torch.Tensor] = None   # fp32 [max S_q, max S_q] query-section bias
    topk_idx: Optional[torch.Tensor] = None  # int32 [total_q, K] key positions per query token
    topk_len: Optional[torch.Tensor] = None  # int32 [total_q] list lengths

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.seqlens_q, default=0))

    @property
    def max_seqlen_k(self) -> int:
        return int(max(self.seqlens_k, default=0))

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def g(self) -> int:
        return self.hq // self.hk

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        return Workload(
            self.name, self.hq, self.hk, self.d, self.b, self.num_blocks,
            list(self.seqlens_q), list(self.seqlens_k), mv(self.q), mv(self.k_cache),
            mv(self.v_cache), mv(self.block_table), mv(self.cu_seqlens_q),
            mv(self.seqused_k), self.scale, self.causal, self.softcap, self.window,
            mv(self.sinks), mv(self.alibi_slopes), dict(self.meta), self.kv_fp8,
            self.k_scale, self.v_scale, mv(self.qq_bias), mv(self.topk_idx), mv(self.topk_len))

    # -- counts used for reporting (no attention arithmetic) ------------------
    def visible_pairs(self) -> int:
        """Number of (query row, key) pairs the masks keep, summed over seqs
        (per query head); with top-k lists, the listed entries that are keys
        of their row."""
        if self.topk_idx is not None:
            return self._listed_keys()
        total = 0
        for sq, sk in zip(self.seqlens_q, self.seqlens_k):
            ctx = sk - sq
            for i in range(sq):
                hi = i + ctx if self.causal else sk - 1
                lo = max(0, i + ctx - self.window + 1) if self.window > 0 else 0
                total += max(0, hi - lo + 1)
        return total

    def _listed_keys(self) -> int:
        idx = self.topk_idx.cpu().to(torch.int64)
        n = self.topk_len.cpu().to(torch.int64)
        total = 0
        t = 0
        for sq, sk in zip(self.seqlens_q, self.seqlens_k):
            ctx = sk - sq
            for i in range(sq):
                row = idx[t, :int(n[t])]
                hi = i + ctx if self.causal else sk - 1
                lo = i + ctx - self.window + 1 if self.window > 0 else 0
                total += int(((row >= max(lo, 0)) & (row <= min(hi, sk - 1))).sum())
                t += 1
        return total

    def kv_keys_read(self) -> int:
        """Keys whose K and V rows the method needs, once per (sequence, kv
        head): the union of the rows' visible ranges -- with a sliding window,
        keys [max(0, ctx - W + 1), S_k) (row 0 reaches furthest back); else
        all S_k keys.  With top-k lists, every listed entry of every token."""
        if self.topk_len is not None:
            return int(self.topk_len.to(torch.int64).sum())
        total = 0
        for sq, sk in zip(self.seqlens_q, self.seqlens_k):
            if sq <= 0:
                continue
            lo = max(0, sk - sq - self.window + 1) if self.window > 0 else 0
            total += max(0, sk - lo)
        return total

    def kv_bytes_read(self) -> int:
        """K and V bytes of the keys in ``kv_keys_read``."""
        return self.kv_keys_read() * self.hk * self.d * (1 if self.kv_fp8 else 2) * 2


def topk_lists(seqlens_q, seqlens_k, k: int, seed: int, *, causal: bool = True,
               ragged: bool = False, junk: float = 0.0):
    """Per query token, up to ``k`` distinct key positions drawn uniformly
    (random order) from the keys it may see: [0, i + ctx] when causal, else
    [0, S_k).  ``ragged`` draws each list's length uniformly in [0, k] (capped
    by the keys available).  ``junk`` replaces that fraction of the entries by
    positions that are not keys of the row: -1, S_k or beyond, and (causal)
    keys past i + ctx.  Unused list slots hold -1.  Returns int32
    ([total_q, k] positions, [total_q] lengths), CPU."""
    g = _gen(seed)
    rows, lens = [], []
    for sq, sk in zip(seqlens_q, seqlens_k):
        ctx = sk - sq
        for i in range(sq):
            avail = (i + ctx + 1) if causal else sk
            n = min(k, avail)
            if ragged:
                n = min(n, int(torch.randint(0, k + 1, (1,), generator=g)))
            row = torch.full((k,), -1, dtype=torch.int32)
            pos = torch.randperm(avail, generator=g)[:n].to(torch.int32)
            if junk > 0 and n > 0:
                bad = torch.rand(n, generator=g) < junk
                kind = torch.randint(0, 3, (n,), generator=g)
                # kind 2: the first key the causal mask hides, else S_k itself
                hidden = i + ctx + 1 if causal and i + ctx + 1 < sk else sk
                alt = torch.where(kind == 0, torch.full_like(pos, -1),
                                  torch.where(kind == 1, torch.full_like(pos, sk + 3),
                                              torch.full_like(pos, hidden)))
                pos = torch.where(bad, alt, pos)
            row[:n] = pos
            rows.append(row)
            lens.append(n)
    idx = torch.stack(rows) if rows else torch.zeros((0, k), dtype=torch.int32)
    return idx, torch.tensor(lens, dtype=torch.int32)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _randint(g, lo, hi, n):
    """n integers uniform in [lo, hi] inclusive."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def build(name: str, hq: int, hk: int, d: int, b: int, seqlens_q, seqlens_k,
          num_blocks: int, scale: float, *, block_ids: Optional[torch.Tensor] = None,
          seed: int = 0, device="cpu", std: float = 1.0, causal: bool = True,
          softcap: float = 0.0, window: int = 0, sinks: bool = False,
          alibi: bool = False, poison: bool = True, bt_pad: int = 0,
          values: bool = True, kv_fp8: bool = False, kv_scale: float = 1.0 / 32,
          qq_bias: bool = False) -> Workload:
    """Assemble a workload from explicit lengths.

    ``block_ids`` (int, len >= sum of blocks needed) fixes the physical blocks
    in table order; by default they are a seeded permutation of the pool.
    """
    seqlens_q = [int(x) for x in seqlens_q]
    seqlens_k = [int(x) for x in seqlens_k]
    n = len(seqlens_q)
    assert len(seqlens_k) == n
    g = _gen(seed)
    nblk = [(sk + b - 1) // b for sk in seqlens_k]
    need = sum(nblk)
    assert need <= num_blocks, (need, num_blocks)
    if block_ids is None:
        block_ids = torch.randperm(num_blocks, generator=g)[:need]
    block_ids = block_ids.to(torch.int64)
    width = max(max(nblk, default=0), 1) + bt_pad
    table = torch.full((n, width), -1, dtype=torch.int32)
    off = 0
    for s in range(n):
        table[s, :nblk[s]] = block_ids[off:off + nblk[s]].to(torch.int32)
        off += nblk[s]
    cu = torch.zeros(n + 1, dtype=torch.int32)
    if n:
        cu[1:] = torch.cumsum(torch.tensor(seqlens_q, dtype=torch.int64), 0).to(torch.int32)
    seqused = torch.tensor(seqlens_k, dtype=torch.int32)
    total_q = sum(seqlens_q)

    dev = torch.device(device)
    vg = torch.Generator(device=dev)
    vg.manual_seed(seed * 7919 + 17)

    def randn(*shape):
        x = torch.randn(*shape, generator=vg, device=dev, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    q = randn(total_q, hq, d) if values else torch.zeros(total_q, hq, d, dtype=torch.bfloat16, device=dev)

    def kv_values(*shape):
        if not kv_fp8:
            return randn(*shape)
        x = torch.randn(*shape, generator=vg, device=dev, dtype=torch.float32)
        x.mul_(std / kv_scale).clamp_(-448.0, 448.0)
        return x.to(torch.float8_e4m3fn).view(torch.uint8)

    if kv_fp8:
        nan = 0x7f
        fill = nan if poison else 0
        k_cache = torch.full((num_blocks, b, hk, d), fill, dtype=torch.uint8, device=dev)
        v_cache = torch.full((num_blocks, b, hk, d), fill, dtype=torch.uint8, device=dev)
    else:
        nan = float("nan")
        fill = nan if poison else 0.0
        k_cache = torch.full((num_blocks, b, hk, d), fill, dtype=torch.bfloat16, device=dev)
        v_cache = torch.full((num_blocks, b, hk, d), fill, dtype=torch.bfloat16, device=dev)
    if values and need:
        ids = block_ids.to(dev)
        k_cache.index_copy_(0, ids, kv_values(need, b, hk, d))
        v_cache.index_copy_(0, ids, kv_values(need, b, hk, d))
    if poison:
        for s in range(n):
            tail = seqlens_k[s] % b
            if nblk[s] and tail:
                last = int(table[s, nblk[s] - 1])
                k_cache[last, tail:] = nan
                v_cache[last, tail:] = nan

    sink_t = torch.randn(hq, generator=g, dtype=torch.float32) if sinks else None
    alibi_t = None
    if alibi:
        alibi_t = torch.tensor([2.0 ** (-8.0 * h / hq) for h in range(1, hq + 1)],
                               dtype=torch.float32)
    qq_t = None
    if qq_bias:
        mq = max(max(seqlens_q, default=1), 1)
        qq_t = torch.randn(mq, mq, generator=g, dtype=torch.float32)
    w = Workload(name, hq, hk, d, b, num_blocks, seqlens_q, seqlens_k, q, k_cache,
                 v_cache, table, cu, seqused, float(scale), causal, float(softcap),
                 int(window), sink_t, alibi_t, {"seed": seed}, bool(kv_fp8),
                 float(kv_scale) if kv_fp8 else 1.0, float(kv_scale) if kv_fp8 else 1.0, qq_t)
    if dev.type != "cpu":
        w.block_table = w.block_table.to(dev)
        w.cu_seqlens_q = w.cu_seqlens_q.to(dev)
        w.seqused_k = w.seqused_k.to(dev)
        if w.sinks is not None:
            w.sinks = w.sinks.to(dev)
        if w.alibi_slopes is not None:
            w.alibi_slopes = w.alibi_slopes.to(dev)
        if w.qq_bias is not None:
            w.qq_bias = w.qq_bias.to(dev)
    return w


def make(name: str, device="cpu", poison: bool = False, values: bool = True) -> Workload:
    """One of the five named benchmark workloads (seed = 1000 + config index)."""
    idx = _CONFIG_INDEX[name]
    seed = 1000 + idx
    g = _gen(seed)
    common = dict(seed=seed, device=device, poison=poison, values=values)
    if name == "tiny":
        return build(name, 4, 1, 64, 16, [128], [128], 32, 1.0 / 8.0, **common)
    if name in ("decode", "decode_fp8", "decode_d64", "decode_d256"):
        sk = _randint(g, 512, 8192, 64)
        d = {"decode_d64": 64, "decode_d256": 256}.get(name, 128)
        return build(name, 32, 8, d, 16, [1] * 64, sk, 40000, 1.0 / math.sqrt(d),
                     kv_fp8=name == "decode_fp8", **common)
    if name == "chunked":
        ctx = _randint(g, 0, 4096, 16)
        sq = _randint(g, 1, 512, 16)
        sk = [c + q for c, q in zip(ctx, sq)]
        return build(name, 32, 8, 128, 32, sq, sk, 4096, 1.0 / math.sqrt(128),
                     softcap=50.0, window=1024, sinks=True, **common)
    if name in ("long_prefill", "long_prefill_shuffled"):
        ids = torch.arange(128) if name == "long_prefill" else torch.randperm(128, generator=g)
        return build(name, 128, 8, 128, 64, [8192], [8192], 128, 1.0 / math.sqrt(128),
                     block_ids=ids, **common)
    if name == "wide_mha_alibi":
        return build(name, 32, 32, 256, 64, [4096] * 8, [4096] * 8, 512,
                     1.0 / math.sqrt(256), std=0.5, alibi=True, **common)
    if name == "decode_topk":
        sk = _randint(g, 4096, 16384, 256)
        w = build(name, 16, 1, 128, 64, [1] * 256, sk, 48000, 1.0 / math.sqrt(128), **common)
        idx, lens = topk_lists(w.seqlens_q, w.seqlens_k, 2048, seed + 1)
        w.topk_idx, w.topk_len = idx.to(w.q.device), lens.to(w.q.device)
        return w
    raise KeyError(name)


def random_small(seed: int, *, num_seqs=3, hq=8, hk=2, d=64, b=16, sq=(1, 40),
                 ctx=(0, 70), causal=True, softcap=0.0, window=0, sinks=False,
                 alibi=False, device="cpu", poison=True, spare_blocks=5,
                 std=1.0, kv_fp8=False, kv_scale=1.0 / 32, qq_bias=False, topk=0,
                 topk_ragged=False, topk_junk=0.0) -> Workload:
    """A small seeded ragged batch for parity sweeps (lengths drawn per seq);
    ``topk`` > 0 attaches per-token key lists of that capacity (``topk_lists``)."""
    g = _gen(seed)
    seqlens_q = _randint(g, sq[0], sq[1], num_seqs)
    ctxs = _randint(g, ctx[0], ctx[1], num_seqs)
    seqlens_k = [q + c for q, c in zip(seqlens_q, ctxs)]
    need = sum((k + b - 1) // b for k in seqlens_k)
    w = build("random_small", hq, hk, d, b, seqlens_q, seqlens_k,
              need + spare_blocks, 1.0 / math.sqrt(d), seed=seed, device=device,
              std=std, causal=causal, softcap=softcap, window=window, sinks=sinks,
              alibi=alibi, poison=poison, bt_pad=1, kv_fp8=kv_fp8, kv_scale=kv_scale,
              qq_bias=qq_bias)
    if topk:
        idx, lens = topk_lists(seqlens_q, seqlens_k, topk, seed + 7919, causal=causal,
                               ragged=topk_ragged, junk=topk_junk)
        w.topk_idx, w.topk_len = idx.to(w.q.device), lens.to(w.q.device)
    return w


def sample_rows(w: Workload, n: int, seed: int = 0) -> torch.Tensor:
    """Row ids (token * H_q + head) for sampled parity checks: the first and last
    token of every sequence at the first and last head, plus n seeded draws."""
    g = _gen(seed)
    ids = set()
    cu = [0]
    for s in w.seqlens_q:
        cu.append(cu[-1] + s)
    for s in range(w.num_seqs):
        if w.seqlens_q[s] == 0:
            continue
        for tok in (cu[s], cu[s + 1] - 1):
            for h in (0, w.hq - 1):
                ids.add(tok * w.hq + h)
    total = w.total_q * w.hq
    if total:
        for x in torch.randint(0, total, (n,), generator=g).tolist():
            ids.add(int(x))
    return torch.tensor(sorted(ids), dtype=torch.int64)
