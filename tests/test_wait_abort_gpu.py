"""The bounded-wait abort path, run on purpose (GPU only).

Every on-chip wait of the kernels gives up after a bounded time; the kernel
then sets UA_DEVERR_TIMEOUT, raises its CTA abort flag, drains the copies and
MMAs it issued, frees its tensor memory and returns, so that the context stays
usable.  The testing hook ua_debug_stall_data_waits makes a kernel's first K/V
data wait wait on a barrier that nothing completes (with a 2 ms bound): the
call must return promptly with the TIMEOUT bit set, and the next normal call
on the same problem must match the fp64 oracle.  (In the CTA-pair kernel
only CTA 0 stalls; the other CTA's waits give up on their normal one-second
bound.)  The drain waits keep their
normal bound, so no CTA leaves with a copy or an MMA in flight."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import binding
from paged_varlen_flash_gb300 import workloads as W
from tests.helpers import max_mean_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_varlen_flash_gb300 import build
    build.build()
    ua.load_library()


CASES = {
    # path, workload: each kernel family that carries the stall point
    "split": (ua.UA_PATH_SPLIT_KV, dict(num_seqs=5, hq=8, hk=2, d=128, b=16, sq=(1, 3), ctx=(100, 900))),
    "decode_tc": (ua.UA_PATH_DECODE_TC, dict(num_seqs=5, hq=16, hk=4, d=128, b=16, sq=(1, 1),
                                             ctx=(100, 2000))),
    "prefill_pair": (ua.UA_PATH_TENSOR_CORE, dict(num_seqs=4, hq=16, hk=2, d=128, b=32, sq=(60, 300),
                                                  ctx=(0, 400), softcap=30.0)),
    # one dense sequence: the one-CTA-per-unit grid form of the same kernel
    "prefill_grid": (ua.UA_PATH_TENSOR_CORE, dict(num_seqs=1, hq=128, hk=16, d=64, b=32, sq=(640, 640),
                                                  ctx=(0, 0))),
    # d = 256: the CTA-pair kernel (CTA 0 stalls; CTA 1's waits run out on
    # their normal bound, so each stalled call takes about a second)
    "prefill_cta2": (ua.UA_PATH_TENSOR_CORE, dict(num_seqs=2, hq=8, hk=4, d=256, b=32, sq=(200, 300),
                                                  ctx=(0, 300))),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bounded_wait_gives_up_and_the_context_stays_usable(name):
    path, kw = CASES[name]
    w = W.random_small(900 + len(name), **kw)
    want = oracle.forward_workload(w)
    wd = w.to("cuda")
    prob = ua.Problem.for_workload(wd, path=path)
    assert binding.ua_debug_stall_data_waits(prob.handle, 1, 2_000_000) == 0
    for _ in range(2):
        t0 = time.time()
        prob.forward_workload(wd)
        code = prob.check_device_error()
        elapsed = time.time() - t0
        assert code & ua.UA_DEVERR_TIMEOUT, code
        assert elapsed < 5.0, elapsed          # the call returned, nothing hung
    # back to normal calls on the same problem and context
    assert binding.ua_debug_stall_data_waits(prob.handle, 0, 0) == 0
    out = prob.forward_workload(wd)
    assert prob.check_device_error() == 0
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    mx, mn = max_mean_abs(got, want)
    assert mx <= 2e-2 and mn <= 2e-3, (mx, mn)
    prob.close()


def test_stall_hook_argument_checks():
    w = W.random_small(950, num_seqs=2, d=64, b=16).to("cuda")
    prob = ua.Problem.for_workload(w)
    assert binding.ua_debug_stall_data_waits(prob.handle, 1, 10) == 1          # below 1 us
    assert binding.ua_debug_stall_data_waits(prob.handle, 1, 2_000_000_000) == 1
    assert binding.ua_debug_stall_data_waits(None, 0, 0) == 1
    assert binding.ua_debug_stall_data_waits(prob.handle, 0, 0) == 0
    prob.close()
