"""fp8 e4m3 KV cache (bf16 Q, one scale per K / V tensor): the decode tensor-core
kernel against the fp64 oracle, through the C ABI (GPU only).

Same acceptance bar as the bf16 path (max-abs <= 2e-2, mean-abs <= 2e-3 against
the unrounded oracle): e4m3 values are exact in the kernel's f16 operands, so
only the P rounding and the fp32 accumulation differ from the oracle."""
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
    # (b, hq, hk, sq range, ctx range, k_scale, v_scale, flags)
    (16, 32, 8, (1, 1), (100, 900), 1 / 32, 1 / 32, {}),
    (32, 8, 8, (1, 1), (0, 300), 1 / 16, 1 / 64, {}),
    (64, 16, 1, (1, 1), (0, 1300), 1 / 32, 1 / 32, {}),
    (16, 8, 2, (1, 4), (0, 700), 0.03, 0.05, dict(softcap=30.0, window=200, sinks=True)),
    (16, 8, 8, (1, 1), (10, 1000), 1 / 32, 1 / 32, dict(alibi=True)),
    (32, 16, 4, (1, 2), (0, 260), 1 / 32, 1 / 32, dict(causal=False)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fp8_decode_matches_oracle(case):
    b, hq, hk, sq, ctx, ks, vs, flags = CASES[case]
    w = W.random_small(700 + case, num_seqs=5, hq=hq, hk=hk, d=128, b=b, sq=sq, ctx=ctx,
                       kv_fp8=True, kv_scale=ks, **flags)
    w.v_scale = vs
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd)
    out = prob.forward_workload(wd)
    assert prob.check_device_error() == 0
    assert prob.last_path().startswith("decode_tc")
    _check(out.float().cpu().numpy(), want)


def test_fp8_decode_workload_sampled_rows():
    w = W.make("decode_fp8", device="cuda", poison=True)
    prob = ua.Problem.for_workload(w)
    out = prob.forward_workload(w)
    assert prob.check_device_error() == 0
    ids = W.sample_rows(w, 400, seed=9)
    want = oracle.forward_workload(w.to("cpu"), row_ids=ids)
    got = out.float().reshape(-1, w.d)[ids.to("cuda")].cpu().numpy()
    _check(got, want)


def test_fp8_cache_equals_bf16_cache_of_the_decoded_values():
    """Power-of-two scales make code * scale exact in bf16: the fp8 call must
    agree with the bf16 decode kernel on the decoded caches to within the
    rounding of P (bf16 there, f16 here)."""
    w = W.random_small(750, num_seqs=4, hq=16, hk=4, d=128, b=16, sq=(1, 1), ctx=(50, 600),
                       kv_fp8=True, kv_scale=1 / 32, poison=False)
    wd = w.to("cuda")
    out8 = ua.Problem.for_workload(wd).forward_workload(wd).float().cpu().numpy()
    w16 = w.to("cuda")
    w16.k_cache = (wd.k_cache.view(torch.float8_e4m3fn).float() * w.k_scale).to(torch.bfloat16)
    w16.v_cache = (wd.v_cache.view(torch.float8_e4m3fn).float() * w.v_scale).to(torch.bfloat16)
    w16.kv_fp8, w16.k_scale, w16.v_scale = False, 1.0, 1.0
    out16 = ua.Problem.for_workload(w16).forward_workload(w16).float().cpu().numpy()
    mx, mn = max_mean_abs(out8, out16)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)


def test_fp8_contract():
    """fp8 caches: bad scales are rejected; paths other than the decode kernel
    and head sizes other than 128 are unsupported; a call shaped for prefill
    is refused before any launch."""
    w = W.random_small(760, num_seqs=2, hq=8, hk=2, d=128, b=16, sq=(1, 1), kv_fp8=True)
    args = (w.hq, w.hk, w.d, w.b, w.num_blocks, 4, w.max_blocks_per_seq, 64,
            ua.UA_FLAG_CAUSAL, w.scale, 0.0, 0)
    with pytest.raises(ua.UAError) as e:
        ua.Problem(*args, ua.UA_PATH_AUTO, ua.UA_DTYPE_FP8_E4M3, 0.0, 1.0)
    assert e.value.status == 1      # UA_ERR_INVALID_ARG
    with pytest.raises(ua.UAError) as e:
        ua.Problem(*args, ua.UA_PATH_SPLIT_KV, ua.UA_DTYPE_FP8_E4M3, 1.0, 1.0)
    assert e.value.status == 2      # UA_ERR_UNSUPPORTED
    with pytest.raises(ua.UAError) as e:
        ua.Problem(w.hq, w.hk, 64, w.b, w.num_blocks, 4, w.max_blocks_per_seq, 64,
                   ua.UA_FLAG_CAUSAL, w.scale, 0.0, 0, ua.UA_PATH_AUTO, ua.UA_DTYPE_FP8_E4M3,
                   1.0, 1.0)
    assert e.value.status == 2
    pw = W.random_small(761, num_seqs=2, hq=8, hk=2, d=128, b=16, sq=(30, 40), kv_fp8=True).to("cuda")
    prob = ua.Problem.for_workload(pw)
    with pytest.raises(ua.UAError) as e:
        prob.forward_workload(pw)
    assert e.value.status == 2
