"""Sparse top-k decode (ua_forward_topk: each query token attends to its own
list of key positions) against the fp64 oracle, through the C ABI (GPU only).

Lists are drawn with ``workloads.topk_lists``: distinct positions in random
order, ragged lengths, and "junk" entries that are not keys of the row (-1,
past S_k, hidden by the causal mask) which both sides must skip.  Unused cache
slots hold NaN, so a skipped entry whose V row reached the output would show."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import workloads as W
from tests.helpers import decode_tag, max_mean_abs, position_tags, scatter_logical, token_of_row

MAX_ABS = 2e-2
MEAN_ABS = 2e-3

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_varlen_flash_gb300 import build
    build.build()
    ua.load_library()


def _check(got, want):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    mx, mn = max_mean_abs(got, want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


CASES = [
    # (b, hq, hk, sq range, ctx range, K, ragged, junk, flags)
    (16, 16, 1, (1, 1), (100, 3000), 2048, False, 0.0, {}),
    (64, 16, 1, (1, 1), (0, 5000), 1000, True, 0.0, {}),
    (32, 32, 8, (1, 3), (10, 2000), 300, True, 0.2, {}),
    (16, 8, 8, (1, 2), (0, 700), 129, True, 0.3, dict(softcap=30.0, sinks=True)),
    (64, 8, 2, (1, 2), (5, 900), 640, False, 0.1, dict(alibi=True, window=400)),
    (16, 16, 4, (1, 2), (0, 500), 64, True, 0.2, dict(causal=False, qq_bias=True)),
    (32, 4, 1, (1, 4), (0, 1200), 256, True, 0.0, dict(qq_bias=True, sinks=True)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_topk_matches_oracle(case):
    b, hq, hk, sq, ctx, K, ragged, junk, flags = CASES[case]
    w = W.random_small(1100 + case, num_seqs=6, hq=hq, hk=hk, d=128, b=b, sq=sq, ctx=ctx,
                       topk=K, topk_ragged=ragged, topk_junk=junk, **flags)
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd)
    out = prob.forward_workload(wd)
    assert prob.check_device_error() == 0
    assert prob.last_path().startswith("topk_tc"), prob.last_path()
    _check(out.float().cpu().numpy(), want)


def test_topk_workload_sampled_rows():
    w = W.make("decode_topk", device="cuda", poison=True)
    prob = ua.Problem.for_workload(w)
    out = prob.forward_workload(w)
    assert prob.check_device_error() == 0
    ids = W.sample_rows(w, 400, seed=11)
    want = oracle.forward_workload(w.to("cpu"), row_ids=ids)
    got = out.float().reshape(-1, w.d)[ids.to("cuda")].cpu().numpy()
    _check(got, want)


def test_topk_bf16_partials_and_split_paths_agree():
    w = W.random_small(1150, num_seqs=3, hq=16, hk=2, d=128, b=16, sq=(1, 2), ctx=(3000, 4000),
                       topk=3000, topk_ragged=True).to("cuda")
    want = oracle.forward_workload(w.to("cpu"))
    for parts in (ua.UA_PARTIALS_F32, ua.UA_PARTIALS_BF16):
        prob = ua.Problem.for_workload(w, split_partials=parts)
        out = prob.forward_workload(w)
        assert prob.check_device_error() == 0
        assert prob.last_path() == "topk_tc+combine"
        _check(out.float().cpu().numpy(), want)


def test_topk_single_entry_returns_the_value_row_bit_exactly():
    """One listed key: its softmax weight is exactly 1, so O is its V row,
    whose position tags are exact in bf16."""
    sq, sk = [1, 2, 1], [300, 77, 1000]
    need = sum((k + 15) // 16 for k in sk)
    w = W.build("tags", 8, 2, 128, 16, sq, sk, need + 4, 128 ** -0.5, seed=1151, bt_pad=1)
    g = torch.Generator().manual_seed(1152)
    scatter_logical(w, [torch.randn(k, 2, 128, generator=g) for k in sk],
                    [position_tags(k, 2, 128) for k in sk])
    rows, lens, picks = [], [], []
    for s, i, ctx in token_of_row(w):
        j = int(torch.randint(0, i + ctx + 1, (1,), generator=g))
        r = torch.full((5,), -1, dtype=torch.int32)
        r[3] = j                       # after three padding entries
        rows.append(r)
        lens.append(5)
        picks.append(j)
    w.topk_idx, w.topk_len = torch.stack(rows), torch.tensor(lens, dtype=torch.int32)
    wd = w.to("cuda")
    out = ua.Problem.for_workload(wd).forward_workload(wd).float().cpu().numpy()
    for tok, j in enumerate(picks):
        for h in range(w.hq):
            assert decode_tag(out[tok, h]) == (j, h // w.g)


def test_topk_empty_and_all_junk_lists_give_zero_rows():
    w = W.random_small(1153, num_seqs=3, hq=8, hk=2, d=128, b=16, sq=(1, 2), ctx=(10, 200),
                       topk=40, sinks=True)
    w.topk_len[0] = 0
    w.topk_idx[1, :] = -1
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd)
    out = prob.forward_workload(wd).float().cpu().numpy()
    assert prob.check_device_error() == 0
    assert np.all(out[0] == 0) and np.all(out[1] == 0)
    _check(out, want)


def test_topk_bad_length_and_bad_block_are_reported():
    w = W.random_small(1154, num_seqs=3, hq=8, hk=2, d=128, b=16, sq=(1, 1), ctx=(100, 300),
                       topk=64)
    # Token 2's list gets a length past its capacity: its rows become 0.
    w.topk_len[2] = 65
    # A key of token 1 sits in a block whose id is out of range: that key is
    # dropped, the rest of its list still counts.
    s1 = 1
    j = int(w.topk_idx[1, 0])
    bad_blk = j // w.b
    w.block_table[s1, bad_blk] = w.num_blocks + 5
    keep = w.topk_idx[1].clone()
    moved = (keep >= bad_blk * w.b) & (keep < (bad_blk + 1) * w.b)
    ref = W.random_small(1154, num_seqs=3, hq=8, hk=2, d=128, b=16, sq=(1, 1), ctx=(100, 300),
                         topk=64)
    ref.topk_idx[1] = torch.where(moved, torch.full_like(keep, -1), keep)
    want = oracle.forward_workload(ref)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd)
    out = prob.forward_workload(wd).float().cpu().numpy()
    err = prob.check_device_error()
    assert err & ua.UA_DEVERR_BOUNDS and err & ua.UA_DEVERR_BLOCK_ID
    assert np.all(out[2] == 0)
    _check(out[:2], want[:2])


def test_topk_contract():
    w = W.random_small(1155, num_seqs=2, hq=8, hk=2, d=128, b=16, sq=(1, 1), ctx=(10, 50),
                       topk=16).to("cuda")
    prob = ua.Problem.for_workload(w)
    flags = ua.flags_of(w.causal)
    args = [prob.handle, w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
            w.seqused_k, w.num_seqs, w.total_q, w.max_seqlen_q, w.max_seqlen_k, w.topk_idx,
            w.topk_len, 16, flags, None, None, torch.empty_like(w.q)]
    assert ua.ua_forward_topk(*args) == 0
    bad = list(args)
    bad[13] = 0
    assert ua.ua_forward_topk(*bad) == 1                       # topk_stride < 1
    bad = list(args)
    bad[11] = None
    assert ua.ua_forward_topk(*bad) == 1                       # no lists
    w64 = W.random_small(1156, d=64, topk=16).to("cuda")
    p64 = ua.Problem.for_workload(w64)
    with pytest.raises(ua.UAError) as e:
        p64.forward_workload(w64)
    assert e.value.status == 2                                  # d = 64
    wg = W.random_small(1157, hq=32, hk=1, d=128, topk=16).to("cuda")
    with pytest.raises(ua.UAError) as e:
        ua.Problem.for_workload(wg).forward_workload(wg)
    assert e.value.status == 2                                  # g = 32 > 16
