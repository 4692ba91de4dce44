"""ua_forward_noalloc: the allocation-free entry point for callers that cannot
call cudaMalloc (memory arenas that own the whole device, stream-capture
regions, plugins handed only the call's tensors).  Its split partials live in
a static device array inside the library instead of a problem workspace.

Checked through the C ABI against ua_forward on the same inputs, on two calls
in a row (the second call finds the first call's partials still in the shared
array), and against the fp64 CPU oracle directly, with the tolerance of the
parity tests.  This file is collected last so that a failure here cannot hide
another test's result."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_flash_gb300 as ua
from paged_varlen_flash_gb300 import binding
from paged_varlen_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_varlen_flash_gb300 import build
    build.build()
    ua.load_library()


def _desc(w, path=0, partials=0):
    flags = ua.flags_of(w.causal, w.softcap, w.alibi_slopes is not None, w.window,
                        w.sinks is not None)
    return binding.ProblemDesc(w.hq, w.hk, w.d, w.b, w.num_blocks, max(1, w.num_seqs),
                               w.max_blocks_per_seq, max(1, w.total_q), 0, flags, w.scale,
                               w.softcap, w.window, path, 0, 1.0, 1.0, partials), flags


def _noalloc(w, out, err=None, path=0, partials=0):
    desc, flags = _desc(w, path, partials)
    return binding.ua_forward_noalloc(desc, w.q, w.k_cache, w.v_cache, w.block_table,
                                 w.cu_seqlens_q, w.seqused_k, w.num_seqs, w.total_q,
                                 w.max_seqlen_q, w.max_seqlen_k, flags, w.sinks,
                                 w.alibi_slopes, out, err)


def _close(a, b):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, (d.max().item(),
                                                                        d.mean().item())


@pytest.mark.parametrize("name", ["decode", "small"])
def test_noalloc_matches_forward_on_two_calls(name):
    if name == "decode":
        w = W.make("decode", device="cuda", poison=True)
    else:
        w = W.random_small(11, num_seqs=4, hq=8, hk=2, d=128, b=32, sq=(1, 3), ctx=(0, 900),
                           softcap=20.0, window=300, sinks=True).to("cuda")
    prob = ua.Problem.for_workload(w)
    ref = prob.forward_workload(w)
    assert prob.check_device_error() == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out1 = torch.full_like(w.q, float("nan"))
    out2 = torch.full_like(w.q, float("nan"))
    assert _noalloc(w, out1, err) == 0
    assert _noalloc(w, out2, err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _close(out1, ref)
    _close(out2, ref)
    assert torch.equal(out1, out2)


def test_noalloc_interleaved_workloads_do_not_leak_state():
    a = W.random_small(21, num_seqs=3, hq=32, hk=8, d=128, b=16, sq=(1, 1),
                       ctx=(2000, 4000)).to("cuda")
    b = W.random_small(22, num_seqs=5, hq=8, hk=8, d=64, b=64, sq=(1, 2),
                       ctx=(100, 3000)).to("cuda")
    ra = ua.Problem.for_workload(a).forward_workload(a)
    rb = ua.Problem.for_workload(b).forward_workload(b)
    oa = torch.empty_like(a.q)
    ob = torch.empty_like(b.q)
    for _ in range(2):
        assert _noalloc(a, oa) == 0
        assert _noalloc(b, ob) == 0
        torch.cuda.synchronize()
        _close(oa, ra)
        _close(ob, rb)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 2048 rows x 64 heads x (256 + 2) floats is 135 MB per segment: far more
    # than the 16 MiB static array.
    w = W.build("big", 64, 8, 256, 64, [1] * 2048, [64] * 2048, 2048, 0.0625, values=False,
                poison=False, device="cuda")
    out = torch.empty_like(w.q)
    assert _noalloc(w, out) == 2   # UA_ERR_UNSUPPORTED, nothing launched
    torch.cuda.synchronize()


def _oracle_close(out, w):
    want = oracle.forward_workload(w.to("cpu"))
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    d = np.abs(got - want)
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())


def test_noalloc_matches_oracle_directly():
    # Decode rows, GQA 4, softcap + window + sinks, NaN in every unused slot.
    w = W.random_small(31, num_seqs=6, hq=16, hk=4, d=128, b=16, sq=(1, 2), ctx=(0, 1500),
                       softcap=30.0, window=700, sinks=True).to("cuda")
    for _ in range(2):
        out = torch.full_like(w.q, float("nan"))
        assert _noalloc(w, out) == 0
        torch.cuda.synchronize()
        _oracle_close(out, w)


def test_noalloc_at_its_largest_accepted_size():
    # 500 rows x 16 heads x (256 + 2) floats = 8.26 MB per segment, just under
    # half the 16 MiB array (the largest per-segment size accepted): exactly
    # two segments fit, and the split planner picks two for this batch.
    # ALiBi and bf16 partials on.
    w = W.random_small(32, num_seqs=1, hq=16, hk=2, d=256, b=64, sq=(500, 500), ctx=(900, 1000),
                       alibi=True).to("cuda")
    out = torch.full_like(w.q, float("nan"))
    assert _noalloc(w, out, partials=ua.UA_PARTIALS_BF16) == 0
    torch.cuda.synchronize()
    _oracle_close(out, w)


def test_noalloc_path_field_is_checked():
    w = W.random_small(33, num_seqs=2, hq=8, hk=2, d=64, b=16, sq=(1, 1), ctx=(10, 50)).to("cuda")
    out = torch.empty_like(w.q)
    assert _noalloc(w, out, path=ua.UA_PATH_SPLIT_KV) == 0
    assert _noalloc(w, out, path=ua.UA_PATH_TENSOR_CORE) == 2   # UA_ERR_UNSUPPORTED
    assert _noalloc(w, out, path=ua.UA_PATH_DECODE_TC) == 2
    assert _noalloc(w, out, path=7) == 1                        # UA_ERR_INVALID_ARG
    torch.cuda.synchronize()


def test_noalloc_captured_in_a_cuda_graph():
    # The use the entry point exists for: one warm-up call, then the call
    # inside a stream capture (no allocation may happen there), replayed;
    # a second replay after Q changed in place reads the new values.
    w = W.random_small(34, num_seqs=4, hq=16, hk=4, d=128, b=16, sq=(1, 2), ctx=(100, 2000),
                       softcap=25.0, sinks=True).to("cuda")
    prob = ua.Problem.for_workload(w)
    ref = prob.forward_workload(w)
    out = torch.full_like(w.q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert _noalloc(w, out, err) == 0
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert _noalloc(w, out, err) == 0
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _close(out, ref)
    g = torch.Generator(device="cpu").manual_seed(35)
    w.q.copy_(torch.randn(w.q.shape, generator=g).to(w.q.dtype))
    ref2 = prob.forward_workload(w)
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _close(out, ref2)
    assert not torch.equal(ref, ref2)
