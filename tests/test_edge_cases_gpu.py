"""Edge cases of the method on the GPU, each against the fp64 CPU oracle and on
every kernel family that can serve the shape (GPU only):

* caches larger than 2 GiB with every used block past the 2 GiB byte offset
  (gfx950 "Unified paged attention on gfx950, from the math up", section 7.2:
  32-bit offsets would read the wrong rows there), checked bit-exactly with
  position tags;
* sink logits of +inf (the row's output is 0) and -inf (the sink drops out)
  (gfx950 page, section 1 step 7; gfx1151 ALGORITHM.md section 6);
* empty sequences (S_q = 0, with S_k = 0 and with S_k > 0) between non-empty
  ones in one batch;
* GQA groups that do not divide the tensor-core tiles (g = 3, 5, 6, 7;
  gfx950 page, section 4 packs the g heads of one KV head into the tile).

Tolerance as in the other parity tests: max-abs <= 2e-2, mean-abs <= 2e-3
against the unrounded fp64 oracle; index work bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import workloads as W
from tests.helpers import decode_tag, max_mean_abs, position_tags, scatter_logical, tag_values, token_of_row

MAX_ABS = 2e-2
MEAN_ABS = 2e-3

pytestmark = pytest.mark.gpu

SPLIT, TC, DEC = ua.UA_PATH_SPLIT_KV, ua.UA_PATH_TENSOR_CORE, ua.UA_PATH_DECODE_TC
PATHS = [SPLIT, TC, DEC]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_varlen_flash_gb300 import build
    build.build()
    ua.load_library()


def serves(w, path):
    """Whether the forced kernel family takes this shape (else the library
    returns UA_ERR_UNSUPPORTED and the case is skipped)."""
    g = w.hq // w.hk
    if path == TC:
        return g <= 128
    if path == DEC:
        return w.d in (64, 128, 256) and g <= 16 and g * w.max_seqlen_q <= 16
    return True


def run(w, path, topk=False):
    """Forward on the GPU through the C ABI; (output on the CPU, error word)."""
    if not serves(w, path) or (topk and not (w.d == 128 and (w.hq // w.hk) <= 16)):
        pytest.skip("shape outside this kernel family")
    wd = w if w.q.is_cuda else w.to("cuda")
    prob = ua.Problem.for_workload(wd, path=path)
    out = prob.forward_workload(wd)
    err = prob.check_device_error()
    got = out.float().cpu()
    prob.close()
    return got, err


def check_close(got, want):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    mx, mn = max_mean_abs(got, want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


# ---------------------------------------------------------------------------
# Caches beyond 2 GiB.
# ---------------------------------------------------------------------------
def tags_workload(hq, hk, d, b, sq, sk, seed, topk=False):
    """A compact CPU workload whose every row has one dominant key (score
    margin 64) and whose V rows spell out their key index and KV head."""
    need = sum((k + b - 1) // b for k in sk)
    w = W.build("tags", hq, hk, d, b, sq, sk, need + 3, 1.0, seed=seed, values=False,
                poison=True, bt_pad=1)
    q = torch.zeros(w.total_q, hq, d)
    kl = [torch.zeros(k, hk, d) for k in sk]
    g = torch.Generator().manual_seed(seed)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        q[tok, :, i % d] = 1.0
        for hkv in range(hk):
            t = int(torch.randint(0, i + ctx + 1, (1,), generator=g))
            kl[s][t, hkv, i % d] = 64.0
    w.q = q.to(torch.bfloat16)
    scatter_logical(w, kl, [position_tags(k, hk, d) for k in sk])
    if topk:
        # every visible key listed, in a random order, plus padding entries
        idx, lens = W.topk_lists(w.seqlens_q, w.seqlens_k, max(sk) + 8, seed + 1)
        w.topk_idx, w.topk_len = idx, lens
    return w


def relocate_past_2gib(w):
    """The same logical K/V on the GPU in a pool whose used blocks all sit past
    the 2 GiB byte offset of each cache (unused blocks hold NaN)."""
    block_bytes = w.b * w.hk * w.d * 2
    first = (2 << 30) // block_bytes + 5
    need = sum((k + w.b - 1) // w.b for k in w.seqlens_k)
    nb = first + need + 4
    dev = torch.device("cuda")
    k = torch.full((nb, w.b, w.hk, w.d), float("nan"), dtype=torch.bfloat16, device=dev)
    v = torch.full_like(k, float("nan"))
    old = w.block_table
    new = torch.full_like(old, -1)
    perm = torch.randperm(need, generator=torch.Generator().manual_seed(9)) + first
    n = 0
    for s in range(w.num_seqs):
        for i in range((w.seqlens_k[s] + w.b - 1) // w.b):
            new[s, i] = int(perm[n])
            k[int(perm[n])] = w.k_cache[int(old[s, i])].to(dev)
            v[int(perm[n])] = w.v_cache[int(old[s, i])].to(dev)
            n += 1
    big = w.to("cuda")
    big.k_cache, big.v_cache, big.num_blocks = k, v, nb
    big.block_table = new.to(dev)
    assert int(new[new >= 0].min()) * block_bytes >= (2 << 30)
    assert k.numel() * 2 > (2 << 30)
    return big


def assert_tags(got, want, w):
    for tok in range(w.total_q):
        for h in range(w.hq):
            exp_tag = decode_tag(want[tok, h])
            row = got[tok, h].numpy()
            assert decode_tag(row) == exp_tag, (tok, h)
            assert tuple(float(x) for x in row[:4]) == tuple(float(x) for x in tag_values(*exp_tag))
            assert np.all(row[4:] == 0)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d,b,hq,hk,sq,sk", [(128, 64, 32, 8, [1, 1, 1], [700, 130, 2000]),
                                             (128, 64, 16, 8, [70, 1], [300, 900]),
                                             (256, 64, 4, 2, [40, 1], [200, 1100])])
def test_cache_beyond_2gib_position_tags_bit_exact(d, b, hq, hk, sq, sk, path):
    w = tags_workload(hq, hk, d, b, sq, sk, seed=17)
    if not serves(w, path):
        pytest.skip("shape outside this kernel family")
    want = oracle.forward_workload(w)
    big = relocate_past_2gib(w)
    got, err = run(big, path)
    assert err == 0
    assert_tags(got, want, w)


def test_topk_cache_beyond_2gib_position_tags_bit_exact():
    # d = 128, one KV head, b = 64: 16 KiB blocks, 2 GiB = 131,072 blocks.
    w = tags_workload(8, 1, 128, 64, [1, 2, 1], [900, 300, 2100], seed=18, topk=True)
    want = oracle.forward_workload(w)
    big = relocate_past_2gib(w)
    got, err = run(big, ua.UA_PATH_AUTO, topk=True)
    assert err == 0
    assert_tags(got, want, w)


# ---------------------------------------------------------------------------
# Infinite sinks.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS + ["topk"])
@pytest.mark.parametrize("d,sq", [(128, (1, 1)), (128, (1, 4)), (64, (20, 90)), (256, (1, 30))])
def test_infinite_sinks(d, sq, path):
    topk = path == "topk"
    w = W.random_small(500 + d + sq[1], num_seqs=4, hq=8, hk=2, d=d, b=16, sq=sq, ctx=(0, 300),
                       sinks=True, softcap=20.0, topk=160 if topk else 0, topk_ragged=topk)
    if topk and (w.d != 128 or w.max_seqlen_q > 4):
        pytest.skip("top-k decode shapes only")
    # heads 0, 3: +inf (output 0); heads 1, 6: -inf (no sink); others finite
    w.sinks[0] = w.sinks[3] = math.inf
    w.sinks[1] = w.sinks[6] = -math.inf
    want = oracle.forward_workload(w)
    got, err = run(w, ua.UA_PATH_AUTO if topk else path, topk=topk)
    assert err == 0
    g = got.numpy()
    assert np.all(g[:, [0, 3], :] == 0)
    check_close(g, want)


# ---------------------------------------------------------------------------
# Empty sequences between non-empty ones.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS + ["topk"])
@pytest.mark.parametrize("shape", ["decode", "prefill"])
def test_empty_sequences_mid_batch(shape, path):
    topk = path == "topk"
    if shape == "decode":
        sq = [1, 0, 2, 0, 1, 0]
        sk = [300, 0, 500, 77, 1, 0]
    else:
        if topk:
            pytest.skip("top-k decode shapes only")
        sq = [40, 0, 130, 0, 1, 7]
        sk = [40, 0, 400, 260, 90, 7]
    need = sum((k + 16 - 1) // 16 for k in sk)
    w = W.build("empty", 8, 2, 128, 16, sq, sk, need + 4, 1.0 / math.sqrt(128), seed=41,
                poison=True, bt_pad=1, sinks=True, softcap=30.0)
    if topk:
        idx, lens = W.topk_lists(sq, sk, 200, 43, ragged=True)
        w.topk_idx, w.topk_len = idx, lens
    want = oracle.forward_workload(w)
    got, err = run(w, ua.UA_PATH_AUTO if topk else path, topk=topk)
    assert err == 0
    check_close(got.numpy(), want)


# ---------------------------------------------------------------------------
# GQA groups that do not divide the tiles.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("hq,hk", [(24, 8), (40, 8), (12, 2), (14, 2)])
@pytest.mark.parametrize("d,sq,fl", [(128, (1, 1), {}), (128, (1, 3), dict(softcap=30.0, sinks=True)),
                                     (64, (30, 150), dict(window=100, sinks=True)),
                                     (128, (40, 300), {}), (256, (20, 140), dict(alibi=True))])
def test_gqa_groups_not_dividing_the_tile(hq, hk, d, sq, fl, path):
    w = W.random_small(600 + hq + d + sq[1], num_seqs=3, hq=hq, hk=hk, d=d, b=32, sq=sq,
                       ctx=(0, 260), **fl)
    want = oracle.forward_workload(w)
    got, err = run(w, path)
    assert err == 0
    check_close(got.numpy(), want)


@pytest.mark.parametrize("hq,hk", [(24, 8), (40, 8), (12, 2)])
def test_gqa_groups_not_dividing_the_tile_topk(hq, hk):
    w = W.random_small(650 + hq, num_seqs=4, hq=hq, hk=hk, d=128, b=16, sq=(1, 1), ctx=(100, 900),
                       topk=300, topk_ragged=True, topk_junk=0.1, sinks=True)
    if (hq // hk) > 16:
        pytest.skip("g > 16")
    want = oracle.forward_workload(w)
    got, err = run(w, ua.UA_PATH_AUTO, topk=True)
    assert err == 0
    check_close(got.numpy(), want)
