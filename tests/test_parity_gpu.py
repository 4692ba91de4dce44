"""CUDA path vs the fp64 CPU oracle, through the C ABI (GPU only).

Tolerance (the acceptance bar for bf16 outputs of N(0,1)-scale inputs):
max-abs error <= 2e-2 and mean-abs error <= 2e-3 against the unrounded fp64
oracle.  Index work (which key, which block, which head) is checked bit-exactly
with position-tag values."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import workloads as W
from tests.helpers import (decode_tag, max_mean_abs, position_tags, scatter_logical, tag_values,
                           token_of_row)

MAX_ABS = 2e-2
MEAN_ABS = 2e-3

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_varlen_flash_gb300 import build
    build.build()
    ua.load_library()


# Every kernel family is checked on every shape it can serve.
PATHS = [ua.UA_PATH_SPLIT_KV, ua.UA_PATH_TENSOR_CORE, ua.UA_PATH_DECODE_TC]


def tc_ok(w):
    return (w.hq // w.hk) <= 128


def dec_ok(w):
    g = w.hq // w.hk
    return w.d in (64, 128, 256) and g <= 16 and g * w.max_seqlen_q <= 16


def run_gpu(w, problem=None, out=None, path=ua.UA_PATH_AUTO):
    if path == ua.UA_PATH_TENSOR_CORE and not tc_ok(w):
        pytest.skip("g > 128")
    if path == ua.UA_PATH_DECODE_TC and not dec_ok(w):
        pytest.skip("not a decode-shaped call for the transposed kernel")
    wd = w.to("cuda")
    prob = problem or ua.Problem.for_workload(wd, path=path)
    res = prob.forward_workload(wd, out=out)
    err = prob.check_device_error()
    return res.float().cpu(), err, prob


def check_close(got, want, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    mx, mn = max_mean_abs(got, want)
    assert mx <= max_abs and mn <= mean_abs, (mx, mn)
    return mx, mn


# ---------------------------------------------------------------------------
# Small ragged sweeps, every row checked.
# ---------------------------------------------------------------------------
SWEEP = [
    # (d, b, hq, hk, sq range, ctx range, flags)
    (64, 16, 4, 1, (1, 1), (0, 300), {}),
    (128, 16, 32, 8, (1, 1), (100, 900), {}),
    (128, 32, 8, 8, (1, 1), (0, 200), {}),
    (256, 64, 4, 4, (1, 1), (0, 500), {}),
    (128, 16, 16, 1, (1, 1), (0, 400), {}),
    (64, 16, 8, 2, (1, 7), (0, 100), {}),
    (128, 32, 8, 2, (1, 40), (0, 130), dict(softcap=50.0, window=64, sinks=True)),
    (128, 16, 8, 2, (1, 3), (0, 700), dict(alibi=True)),
    (64, 64, 4, 2, (5, 30), (0, 90), dict(causal=False)),
    (256, 32, 2, 1, (1, 2), (0, 300), dict(sinks=True, softcap=5.0)),
    (64, 16, 4, 4, (1, 1), (0, 50), dict(window=1)),
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", range(len(SWEEP)))
def test_small_sweep_matches_oracle(case, path):
    d, b, hq, hk, sq, ctx, fl = SWEEP[case]
    w = W.random_small(100 + case, num_seqs=5, hq=hq, hk=hk, d=d, b=b, sq=sq, ctx=ctx, **fl)
    want = oracle.forward_workload(w)
    got, err, _ = run_gpu(w, path=path)
    assert err == 0
    check_close(got, want)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d,b,g,sq", [(64, 16, 4, 128), (128, 32, 4, 300), (128, 64, 16, 40),
                                      (256, 64, 1, 128), (128, 16, 8, 1), (64, 32, 2, 3)])
def test_prefill_shapes_match_oracle(d, b, g, sq, path):
    w = W.random_small(200 + d + b + g, num_seqs=3, hq=2 * g, hk=2, d=d, b=b, sq=(sq // 2 + 1, sq),
                       ctx=(0, 100))
    want = oracle.forward_workload(w)
    got, err, _ = run_gpu(w, path=path)
    assert err == 0
    check_close(got, want)


# ---------------------------------------------------------------------------
# The five benchmark workloads.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS)
def test_tiny_config_full(path):
    w = W.make("tiny", poison=True)
    want = oracle.forward_workload(w)
    got, err, prob = run_gpu(w, path=path)
    assert err == 0
    check_close(got, want)


@pytest.mark.parametrize("path", [ua.UA_PATH_AUTO] + PATHS)
@pytest.mark.parametrize("name", ["decode", "chunked", "long_prefill", "wide_mha_alibi"])
def test_config_sampled_rows(name, path):
    if path == ua.UA_PATH_SPLIT_KV and name in ("long_prefill", "wide_mha_alibi"):
        pytest.skip("CUDA-core path on 2 TFLOP workloads: covered by the smaller prefill shapes")
    if path == ua.UA_PATH_DECODE_TC and name != "decode":
        pytest.skip("not a decode-shaped workload")
    w = W.make(name, device="cuda", poison=(name != "long_prefill"))
    prob = ua.Problem.for_workload(w, path=path)
    out = prob.forward_workload(w)
    assert prob.check_device_error() == 0
    ids = W.sample_rows(w, 400, seed=7)
    want = oracle.forward_workload(w.to("cpu"), row_ids=ids)
    got = out.float().reshape(-1, w.d)[ids.to("cuda")].cpu().numpy()
    check_close(got, want)


def test_long_prefill_shuffled_table_bit_identical():
    a = W.make("long_prefill", device="cuda")
    b = W.make("long_prefill_shuffled", device="cuda", values=False)
    # Same logical K/V behind a shuffled table: move every block to its new home.
    ids = b.block_table[0].long()
    b.k_cache = torch.empty_like(a.k_cache)
    b.v_cache = torch.empty_like(a.v_cache)
    b.k_cache[ids] = a.k_cache[a.block_table[0].long()]
    b.v_cache[ids] = a.v_cache[a.block_table[0].long()]
    b.q = a.q
    pa = ua.Problem.for_workload(a)
    oa = pa.forward_workload(a)
    ob = pa.forward_workload(b)
    assert pa.check_device_error() == 0
    assert torch.equal(oa, ob)


# ---------------------------------------------------------------------------
# Bit-exact index work: one dominant key per (row, kv head) makes the output
# equal to that key's position-tag row.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("d,b,hq,hk,sq,sk", [(64, 16, 8, 2, [7, 30, 1], [40, 30, 77]),
                                             (128, 16, 32, 8, [1, 1, 1], [300, 513, 17]),
                                             (128, 64, 16, 4, [60, 2], [60, 700]),
                                             (256, 32, 4, 4, [33, 1], [90, 2000]),
                                             # full d = 256 tiles (the output goes out by
                                             # TMA from shared memory): g = 1 and g = 2
                                             (256, 64, 4, 4, [256], [300]),
                                             (256, 16, 8, 4, [128, 3], [128, 40])])
def test_position_tags_bit_exact(d, b, hq, hk, sq, sk, path):
    need = sum((k + b - 1) // b for k in sk)
    w = W.build("tags", hq, hk, d, b, sq, sk, need + 7, 1.0, seed=5, values=False, poison=True,
                bt_pad=2)
    q = torch.zeros(w.total_q, w.hq, w.d)
    kl = [torch.zeros(k, w.hk, w.d) for k in sk]
    g = torch.Generator().manual_seed(3)
    targets = {}
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        q[tok, :, i % d] = 1.0
        for hkv in range(w.hk):
            t = int(torch.randint(0, i + ctx + 1, (1,), generator=g))
            # avoid two rows of one sequence sharing a query direction but
            # wanting different keys
            targets[(tok, hkv)] = t
            kl[s][t, hkv, i % d] = 64.0
    w.q = q.to(torch.bfloat16)
    scatter_logical(w, kl, [position_tags(k, w.hk, w.d) for k in sk])
    got, err, _ = run_gpu(w, path=path)
    assert err == 0
    want = oracle.forward_workload(w)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        for h in range(w.hq):
            exp_tag = decode_tag(want[tok, h])
            assert decode_tag(got[tok, h].numpy()) == exp_tag
            row = got[tok, h].numpy()
            assert tuple(float(x) for x in row[:4]) == tuple(float(x) for x in tag_values(*exp_tag))
            assert np.all(row[4:] == 0)


@pytest.mark.parametrize("path", PATHS)
def test_block_permutation_bit_identical_on_gpu(path):
    w = W.random_small(300, num_seqs=4, hq=8, hk=2, d=128, b=16, sq=(1, 20), ctx=(0, 400),
                       softcap=30.0, sinks=True)
    a, err, _ = run_gpu(w, path=path)
    g = torch.Generator().manual_seed(1)
    perm = torch.randperm(w.num_blocks, generator=g)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt = w.block_table.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    w.k_cache, w.v_cache, w.block_table = k2, v2, bt
    b, err2, _ = run_gpu(w, path=path)
    assert err == 0 and err2 == 0
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden) on the GPU.  bf16 output
# rounding is relative, so the bound scales with |expected|.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS)
def test_golden_examples_on_gpu(path):
    from tests.test_oracle_pins import golden_cases, golden_workload
    for case in golden_cases():
        w, expected = golden_workload(case)
        if w.sinks is not None:
            w.sinks = w.sinks.float()
        if w.alibi_slopes is not None:
            w.alibi_slopes = w.alibi_slopes.float()
        got, err, _ = run_gpu(w, path=path)
        assert err == 0, case["name"]
        tol = MAX_ABS * np.maximum(1.0, np.abs(expected))
        assert np.all(np.abs(got.numpy() - expected) <= tol), case["name"]


# ---------------------------------------------------------------------------
# Errors: host-visible contract violations launch nothing; malformed metadata
# is reported through the device error word without a trap.
# ---------------------------------------------------------------------------
def test_host_contract_violations():
    w = W.random_small(400, num_seqs=2, d=64, b=16).to("cuda")
    prob = ua.Problem.for_workload(w)
    out = torch.empty_like(w.q)
    args = [w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k, w.num_seqs,
            w.total_q, w.max_seqlen_q, w.max_seqlen_k]
    fl = ua.UA_FLAG_CAUSAL
    # sinks pointer without the flag, and the flag without a pointer
    sinks = torch.zeros(w.hq, device="cuda")
    assert ua.ua_forward(prob.handle, *args, fl, sinks, None, out) == 1
    assert ua.ua_forward(prob.handle, *args, fl | ua.UA_FLAG_SINKS, None, None, out) == 1
    # flags outside the problem's set
    assert ua.ua_forward(prob.handle, *args, fl | ua.UA_FLAG_ALIBI, None, sinks, out) == 1
    # too many sequences / rows
    bad = list(args)
    bad[6] = w.num_seqs + 100
    assert ua.ua_forward(prob.handle, *bad, fl, None, None, out) == 1
    # misaligned output
    flat = torch.empty(out.numel() + 8, dtype=torch.bfloat16, device="cuda")
    assert ua.ua_forward(prob.handle, *args, fl, None, None, flat[1:]) == 1
    assert prob.check_device_error() == 0


@pytest.mark.parametrize("path", PATHS)
def test_device_reports_bad_block_id_and_short_context(path):
    w = W.random_small(401, num_seqs=3, hq=8, hk=2, d=128, b=16, sq=(1, 1), ctx=(40, 60),
                       poison=False)
    ref = oracle.forward_workload(w)
    # Sequence 1 gets an out-of-range block id; sequence 2 claims fewer keys than queries.
    bad = w.to("cpu")
    bad.block_table = w.block_table.clone()
    bad.block_table[1, 0] = w.num_blocks + 5
    wd = bad.to("cuda")
    prob = ua.Problem.for_workload(wd, path=path)
    out = prob.forward_workload(wd)
    code = prob.check_device_error()
    assert code & ua.UA_DEVERR_BLOCK_ID
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    check_close(got[0], ref[0])          # well-formed sequence unaffected
    check_close(got[2], ref[2])
    assert prob.check_device_error() == 0  # cleared by the previous read

    # Sequence 1 now claims fewer keys (0) than its query rows (1).
    short = w.to("cpu")
    short.block_table = w.block_table.clone()
    short.seqused_k = w.seqused_k.clone()
    short.seqused_k[1] = 0
    wd = short.to("cuda")
    out = prob.forward_workload(wd)
    code = prob.check_device_error()
    assert code & ua.UA_DEVERR_CONTEXT
    got = out.float().cpu().numpy()
    assert np.all(got[1] == 0)
    check_close(got[0], ref[0])
    check_close(got[2], ref[2])


def test_host_buffer_entry_point_matches_device_entry_point():
    w = W.make("decode", device="cuda")
    prob = ua.Problem.for_workload(w)
    dev = prob.forward_workload(w)
    flags = ua.flags_of(w.causal, w.softcap, False, w.window, False)
    q_h = w.q.cpu().pin_memory()
    out_h = torch.empty_like(q_h).pin_memory()
    st = ua.ua_forward_host(prob.handle, q_h, w.k_cache, w.v_cache, w.block_table.cpu(),
                            w.cu_seqlens_q.cpu(), w.seqused_k.cpu(), w.num_seqs, w.total_q,
                            w.max_seqlen_q, w.max_seqlen_k, flags, None, None, out_h)
    assert st == 0
    assert prob.check_device_error() == 0
    assert torch.equal(out_h, dev.cpu())


# ---------------------------------------------------------------------------
# The two forms of the d <= 128 tensor-core prefill: dense batches (the padded
# grid is nearly all real units and fills the GPU twice) run one CTA per unit
# over the grid; ragged ones run persistent CTAs over the planner's
# longest-first list.  Both are checked against the oracle and bit-exactly
# on position tags, and each test asserts which form ran.
# ---------------------------------------------------------------------------
DENSE = dict(num_seqs=1, hq=128, hk=16, d=64, b=32, sq=(640, 640), ctx=(0, 0))


@pytest.mark.parametrize("fl", [{}, dict(softcap=30.0, window=200, sinks=True), dict(alibi=True)])
def test_dense_grid_form_matches_oracle(fl):
    w = W.random_small(710, **DENSE, **fl)
    want = oracle.forward_workload(w)
    got, err, prob = run_gpu(w, path=ua.UA_PATH_TENSOR_CORE)
    assert prob.last_path() == "tensor_core_grid"
    assert err == 0
    check_close(got, want)


def test_ragged_batch_takes_the_persistent_form():
    w = W.random_small(711, num_seqs=6, hq=8, hk=2, d=128, b=16, sq=(1, 300), ctx=(0, 500),
                       softcap=20.0)
    want = oracle.forward_workload(w)
    got, err, prob = run_gpu(w, path=ua.UA_PATH_TENSOR_CORE)
    assert prob.last_path().startswith("tensor_core_pair")
    assert err == 0
    check_close(got, want)


def test_dense_grid_form_position_tags_bit_exact():
    sq = sk = [640]
    d, b, hq, hk = 64, 32, 128, 16
    need = sum((k + b - 1) // b for k in sk)
    w = W.build("tags", hq, hk, d, b, sq, sk, need + 3, 1.0, seed=12, values=False, poison=True,
                bt_pad=1)
    q = torch.zeros(w.total_q, hq, d)
    kl = [torch.zeros(k, hk, d) for k in sk]
    g = torch.Generator().manual_seed(13)
    # S_q > d: rows i and i + d share the query direction i mod d, so rows
    # sharing a direction share one target key, drawn from the keys the first
    # of them (position i mod d, ctx = 0) already sees.
    target = [[int(torch.randint(0, a + 1, (1,), generator=g)) for a in range(d)] for _ in range(hk)]
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        q[tok, :, i % d] = 1.0
        for hkv in range(hk):
            kl[s][target[hkv][i % d], hkv, i % d] = 64.0
    w.q = q.to(torch.bfloat16)
    scatter_logical(w, kl, [position_tags(k, hk, d) for k in sk])
    got, err, prob = run_gpu(w, path=ua.UA_PATH_TENSOR_CORE)
    assert prob.last_path() == "tensor_core_grid"
    assert err == 0
    want = oracle.forward_workload(w)
    for tok in range(w.total_q):
        for h in range(hq):
            exp_tag = decode_tag(want[tok, h])
            assert exp_tag == (target[h // (hq // hk)][tok % d], h // (hq // hk))
            row = got[tok, h].numpy()
            assert decode_tag(row) == exp_tag
            assert tuple(float(x) for x in row[:4]) == tuple(float(x) for x in tag_values(*exp_tag))
            assert np.all(row[4:] == 0)
