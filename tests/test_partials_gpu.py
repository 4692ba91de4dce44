"""bf16 split partials (UA_PARTIALS_BF16): every kernel's KV-split mode writes
its per-segment o in bf16 and the combine kernel reads it back; the result
stays within the acceptance bar of the fp64 oracle and close to the fp32
partials' result (GPU only)."""
import numpy as np
import pytest

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


CASES = [
    # (path, expected path name, d, b, hq, hk, seqlens_q, seqlens_k, extra)
    (ua.UA_PATH_DECODE_TC, "decode_tc+combine", 128, 16, 8, 2, [1, 1], [3900, 3100], {}),
    (ua.UA_PATH_DECODE_TC, "decode_tc+combine", 128, 32, 16, 4, [2, 4], [2600, 4000],
     dict(softcap=30.0, sinks=True)),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_pair+combine", 128, 32, 8, 2, [200], [3200], {}),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_pair+combine", 64, 16, 4, 4, [150], [2500],
     dict(alibi=True, sinks=True)),
    (ua.UA_PATH_TENSOR_CORE, "tensor_core_cta2+combine", 256, 64, 4, 2, [150], [3000], {}),
    (ua.UA_PATH_SPLIT_KV, "split_kv+combine", 128, 16, 8, 2, [1, 3], [3000, 2000],
     dict(window=700)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_bf16_partials_match_oracle_and_fp32_partials(case):
    path, name, d, b, hq, hk, sq, sk, extra = CASES[case]
    need = sum((k + b - 1) // b for k in sk)
    w = W.build("partials", hq, hk, d, b, sq, sk, need + 3, d ** -0.5, seed=900 + case,
                **extra)
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    outs = {}
    for parts in (ua.UA_PARTIALS_F32, ua.UA_PARTIALS_BF16):
        prob = ua.Problem.for_workload(wd, path=path, split_partials=parts)
        outs[parts] = prob.forward_workload(wd).float().cpu().numpy()
        assert prob.check_device_error() == 0
        assert prob.last_path() == name, prob.last_path()
    got = np.asarray(outs[ua.UA_PARTIALS_BF16], dtype=np.float64)
    assert np.all(np.isfinite(got))
    mx, mn = max_mean_abs(got, want)
    assert mx <= MAX_ABS and mn <= MEAN_ABS, (mx, mn)
    # One extra bf16 rounding of each partial before the merge: the two
    # results differ by a few bf16 ulps of the output at most.
    diff = np.abs(outs[ua.UA_PARTIALS_BF16] - outs[ua.UA_PARTIALS_F32])
    assert diff.max() <= 2e-2 and diff.mean() <= 1e-3, (diff.max(), diff.mean())


def test_unknown_partials_type_is_rejected():
    w = W.random_small(950, d=128).to("cuda")
    with pytest.raises(ua.UAError):
        ua.Problem.for_workload(w, split_partials=2)
