"""Query-query bias (score chain step 4: B[i][j - ctx] added to the scores of the
query-section keys, after softcap and ALiBi, before the masks) on every kernel
path against the fp64 oracle, through the C ABI (GPU only).

The bias is N(0, 1), so a wrong index (transposed B, a missing ctx shift, the
bias on context keys) moves outputs by far more than the tolerance."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import workloads as W
from tests.helpers import max_mean_abs

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
    # (path, path-name prefix, d, b, hq, hk, sq range, ctx range, extra flags)
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_pair", 128, 16, 8, 2, (60, 300), (0, 200), {}),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_pair", 64, 32, 4, 4, (100, 300), (0, 0),
     dict(causal=False)),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_pair", 128, 64, 16, 2, (30, 200), (0, 400),
     dict(softcap=30.0, alibi=True, window=150, sinks=True)),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_cta2", 256, 32, 4, 2, (50, 260), (0, 150),
     dict(alibi=True)),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_cta2", 256, 16, 2, 1, (100, 200), (0, 60),
     dict(causal=False, softcap=20.0)),
    (ua.UA_PATH_SPLIT_KV, "split_kv", 128, 16, 8, 2, (1, 70), (0, 300), {}),
    (ua.UA_PATH_SPLIT_KV, "split_kv", 64, 32, 6, 3, (1, 40), (0, 500),
     dict(causal=False, softcap=30.0, sinks=True)),
    (ua.UA_PATH_DECODE_TC, "decode_tc", 128, 16, 16, 4, (1, 4), (0, 900), {}),
    (ua.UA_PATH_DECODE_TC, "decode_tc", 128, 32, 8, 4, (1, 2), (5, 700),
     dict(causal=False, alibi=True)),
    (ua.UA_PATH_DECODE_TC, "decode_tc", 128, 64, 16, 8, (1, 2), (0, 400),
     dict(window=100, softcap=30.0)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_qq_bias_matches_oracle(case):
    path, name, d, b, hq, hk, sq, ctx, flags = CASES[case]
    w = W.random_small(800 + case, num_seqs=4, hq=hq, hk=hk, d=d, b=b, sq=sq, ctx=ctx,
                       qq_bias=True, **flags)
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd, path=path)
    out = prob.forward_workload(wd)
    assert prob.check_device_error() == 0
    assert prob.last_path().startswith(name), prob.last_path()
    _check(out.float().cpu().numpy(), want)


def test_qq_bias_on_an_fp8_cache():
    w = W.random_small(830, num_seqs=5, hq=16, hk=4, d=128, b=16, sq=(1, 3), ctx=(0, 600),
                       kv_fp8=True, kv_scale=1 / 32, qq_bias=True, alibi=True)
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd)
    out = prob.forward_workload(wd)
    assert prob.check_device_error() == 0
    assert prob.last_path().startswith("decode_tc")
    _check(out.float().cpu().numpy(), want)


def test_qq_bias_row_stride_and_a_larger_matrix():
    """B is read through its row stride, and only its leading S_q x S_q corner
    matters: a bigger matrix whose extra rows and columns are huge gives the
    oracle's result on the corner."""
    w = W.random_small(831, num_seqs=3, hq=8, hk=2, d=128, b=16, sq=(40, 90), ctx=(0, 100),
                       qq_bias=True)
    want = oracle.forward_workload(w)
    n = w.qq_bias.shape[0]
    big = torch.full((n + 7, n + 19), 1e4, dtype=torch.float32)
    big[:n, :n] = w.qq_bias
    wd = w.to("cuda")
    for path in (ua.UA_PATH_TENSOR_CORE, ua.UA_PATH_SPLIT_KV):
        prob = ua.Problem.for_workload(wd, path=path)
        wd.qq_bias = big.to("cuda")[:, :]
        out = prob.forward_workload(wd)
        assert prob.check_device_error() == 0
        _check(out.float().cpu().numpy(), want)


def test_qq_bias_workload_scale_prefill_sampled_rows():
    """A long causal prefill (several 128-key tiles per row) on the pair kernel,
    checked on sampled rows."""
    w = W.build("qq_prefill", 16, 4, 128, 32, [1500, 900, 2000], [1500, 1400, 2600], 400,
                128 ** -0.5, seed=832, device="cuda", qq_bias=True)
    prob = ua.Problem.for_workload(w)
    out = prob.forward_workload(w)
    assert prob.check_device_error() == 0
    assert prob.last_path().startswith("tensor_core_pair")
    ids = W.sample_rows(w, 300, seed=4)
    want = oracle.forward_workload(w.to("cpu"), row_ids=ids)
    got = out.float().reshape(-1, w.d)[ids.to("cuda")].cpu().numpy()
    _check(got, want)


def test_qq_flag_without_a_bias_or_with_too_small_a_bias_is_rejected():
    w = W.random_small(833, num_seqs=2, hq=8, hk=2, d=128, b=16, sq=(20, 30), ctx=(0, 10),
                       qq_bias=True).to("cuda")
    prob = ua.Problem.for_workload(w)
    flags = ua.flags_of(w.causal, qq_bias=True)
    args = (prob.handle, w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
            w.seqused_k, w.num_seqs, w.total_q, w.max_seqlen_q, w.max_seqlen_k, flags, None,
            None, torch.empty_like(w.q))
    assert ua.ua_forward(*args) == 1                      # no bias bound yet
    small = torch.zeros(w.max_seqlen_q - 1, w.max_seqlen_q - 1, device="cuda")
    prob.set_qq_bias(small)
    assert ua.ua_forward(*args) == 1                      # max_seqlen_q > n
    assert ua.ua_set_qq_bias(prob.handle, small, 4, 3) == 1   # row_stride < n
    prob.set_qq_bias(w.qq_bias)
    assert ua.ua_forward(*args) == 0
    plain = ua.Problem.for_workload(W.random_small(834, d=128).to("cuda"))
    with pytest.raises(ua.UAError):
        plain.set_qq_bias(w.qq_bias)                      # problem created without the flag
