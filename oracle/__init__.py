"""fp64 CPU oracle for unified paged varlen attention (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
(``paged_varlen_flash_gb300``) and imports nothing from it.

The arithmetic lives in ``ua_oracle.c`` (see its header for the definition it
evaluates and the passages it follows).  This module only marshals numpy /
torch CPU arrays into that library.

Parity status: every term of the definition is pinned by the closed-form and
invariant tests in ``tests/test_oracle_pins.py`` (the e4m3 decoder of the fp8
KV cache against PyTorch's float8_e4m3fn conversion for all 256 codes, and
fp8 attention against the same attention on the decoded values; the sparse
top-k mode against the dense definition on full and permuted lists); the one
part left unpinned is the absolute accuracy of libm's ``tanh`` inside the
softcap term, which is far below any tolerance used against the GPU.
"""
import ctypes
import os

import numpy as np

from . import build as _build

ERRORS = {
    0: "ok",
    -1: "malformed arguments",
    -2: "seqused_k < S_q for some sequence",
    -3: "block id outside [0, num_blocks)",
    -4: "cu_seqlens_q is not non-decreasing from 0",
    -5: "out of memory",
}

_lib = None


class OracleError(RuntimeError):
    def __init__(self, code):
        super().__init__("oracle: %s (code %d)" % (ERRORS.get(code, "?"), code))
        self.code = code


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        common = [ctypes.c_int32] * 5 + [ctypes.c_int64] + [ctypes.c_void_p] * 4 + [
            ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_int32, ctypes.c_double, ctypes.c_int32, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_double, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.ua_oracle_forward.argtypes = common + [ctypes.c_void_p, ctypes.c_int32]
        lib.ua_oracle_forward.restype = ctypes.c_int
        lib.ua_oracle_rows.argtypes = common + [ctypes.c_void_p, ctypes.c_int64,
                                                ctypes.c_void_p, ctypes.c_int32]
        lib.ua_oracle_rows.restype = ctypes.c_int
        lib.ua_oracle_row_weights.argtypes = common + [ctypes.c_int64, ctypes.c_int32,
                                                       ctypes.c_void_p, ctypes.c_void_p]
        lib.ua_oracle_row_weights.restype = ctypes.c_int
        lib.ua_oracle_e4m3.argtypes = [ctypes.c_uint32]
        lib.ua_oracle_e4m3.restype = ctypes.c_double
        _lib = lib
    return _lib


def default_threads():
    """Every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _bf16_bits(t):
    """A torch bf16 tensor or a uint16 array -> contiguous uint16 numpy array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


def _kv_bits(t):
    """A K/V cache -> (contiguous numpy codes, is_fp8): bf16 as uint16 bit
    patterns, fp8 e4m3 (torch float8_e4m3fn, or a uint8 array of codes) as uint8."""
    if isinstance(t, np.ndarray):
        if t.dtype == np.uint8:
            return np.ascontiguousarray(t), True
        return _bf16_bits(t), False
    import torch
    if t.dtype == torch.float8_e4m3fn:
        return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.uint8).numpy()), True
    if t.dtype == torch.uint8:
        return np.ascontiguousarray(t.detach().cpu().contiguous().numpy()), True
    return _bf16_bits(t), False


def e4m3_value(code):
    """The oracle's value of one e4m3 code (0..255)."""
    return float(_load().ua_oracle_e4m3(int(code)))


def _i32(t):
    if not isinstance(t, np.ndarray):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(t, dtype=np.int32)


def _f64_or_none(t):
    if t is None:
        return None
    if not isinstance(t, np.ndarray):
        t = t.detach().cpu().numpy()
    return np.ascontiguousarray(t, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class _Args:
    """Keeps the marshalled arrays alive for the duration of a call."""

    def __init__(self, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                 scale, causal=True, softcap=0.0, window=0, alibi_slopes=None,
                 sinks=None, k_scale=1.0, v_scale=1.0, qq_bias=None, topk_idx=None,
                 topk_len=None):
        self.q = _bf16_bits(q)
        self.topk_idx = self.topk_len = None
        self.topk_stride = 0
        if topk_idx is not None:
            self.topk_idx = _i32(topk_idx)
            assert self.topk_idx.ndim == 2
            self.topk_stride = self.topk_idx.shape[1]
            self.topk_len = _i32(topk_len)
            assert self.topk_len.shape == (self.topk_idx.shape[0],)
        self.qq = _f64_or_none(qq_bias)
        if self.qq is not None:
            assert self.qq.ndim == 2
            self.qq = np.ascontiguousarray(self.qq)
        self.k, fp8_k = _kv_bits(k_cache)
        self.v, fp8_v = _kv_bits(v_cache)
        assert fp8_k == fp8_v, "K and V caches must share a dtype"
        self.kv_fp8 = 1 if fp8_k else 0
        self.k_scale = float(k_scale)
        self.v_scale = float(v_scale)
        self.bt = _i32(block_table)
        self.cu = _i32(cu_seqlens_q)
        self.su = _i32(seqused_k)
        self.alibi = _f64_or_none(alibi_slopes)
        self.sinks = _f64_or_none(sinks)
        assert self.q.ndim == 3 and self.k.ndim == 4 and self.v.shape == self.k.shape
        self.total_q, self.hq, self.d = self.q.shape
        self.num_blocks, self.b, self.hk, dk = self.k.shape
        assert dk == self.d
        self.num_seqs = self.su.shape[0]
        assert self.cu.shape[0] == self.num_seqs + 1
        self.bt = self.bt.reshape(self.num_seqs, -1) if self.num_seqs else self.bt.reshape(0, max(1, self.bt.size))
        self.bt_stride = self.bt.shape[1] if self.bt.ndim == 2 else 1
        self.scale = float(scale)
        self.causal = 1 if causal else 0
        self.softcap = float(softcap or 0.0)
        self.window = int(window or 0)

    def head(self):
        return [self.num_seqs, self.hq, self.hk, self.d, self.b, self.num_blocks,
                _ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.bt), self.bt_stride,
                _ptr(self.cu), _ptr(self.su), self.scale, self.causal, self.softcap,
                self.window, _ptr(self.alibi), _ptr(self.sinks), self.kv_fp8,
                self.k_scale, self.v_scale, _ptr(self.qq),
                self.qq.shape[1] if self.qq is not None else 0,
                _ptr(self.topk_idx), _ptr(self.topk_len), self.topk_stride]


def forward(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, scale,
            causal=True, softcap=0.0, window=0, alibi_slopes=None, sinks=None,
            nthreads=None, k_scale=1.0, v_scale=1.0, qq_bias=None, topk_idx=None,
            topk_len=None):
    """All output rows, fp64 numpy [total_q, H_q, d].  fp8 caches are e4m3
    codes scaled by k_scale / v_scale; qq_bias [>= S_q, stride] is the
    query-section bias shared by all sequences and heads; topk_idx
    [total_q, K] with topk_len [total_q] gives each query token its own key
    list (sparse top-k mode; entries outside [0, S_k) are padding)."""
    a = _Args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, scale,
              causal, softcap, window, alibi_slopes, sinks, k_scale, v_scale, qq_bias,
              topk_idx, topk_len)
    out = np.zeros((a.total_q, a.hq, a.d), dtype=np.float64)
    rc = _load().ua_oracle_forward(*a.head(), _ptr(out),
                                   nthreads or default_threads())
    if rc != 0:
        raise OracleError(rc)
    return out


def rows(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, scale, row_ids,
         causal=True, softcap=0.0, window=0, alibi_slopes=None, sinks=None,
         nthreads=None, k_scale=1.0, v_scale=1.0, qq_bias=None, topk_idx=None,
         topk_len=None):
    """Selected output rows (row id = token * H_q + head), fp64 numpy [n, d]."""
    a = _Args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, scale,
              causal, softcap, window, alibi_slopes, sinks, k_scale, v_scale, qq_bias,
              topk_idx, topk_len)
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64))
    out = np.zeros((ids.shape[0], a.d), dtype=np.float64)
    rc = _load().ua_oracle_rows(*a.head(), _ptr(ids), ids.shape[0], _ptr(out),
                                nthreads or default_threads())
    if rc != 0:
        raise OracleError(rc)
    return out


def row_weights(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, scale,
                token, head, causal=True, softcap=0.0, window=0, alibi_slopes=None,
                sinks=None, k_scale=1.0, v_scale=1.0, qq_bias=None, topk_idx=None,
                topk_len=None):
    """(weights [n + 1] with the sink's share last, O_i [d]) for one row; n is
    S_k, or the row's top-k list length in the sparse mode."""
    a = _Args(q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, scale,
              causal, softcap, window, alibi_slopes, sinks, k_scale, v_scale, qq_bias,
              topk_idx, topk_len)
    cu = a.cu
    s = int(np.searchsorted(cu, token, side="right") - 1)
    while s + 1 < len(cu) and cu[s + 1] <= token:
        s += 1
    n = int(a.su[s]) if a.topk_idx is None else int(a.topk_len[token])
    w = np.zeros(n + 1, dtype=np.float64)
    o = np.zeros(a.d, dtype=np.float64)
    rc = _load().ua_oracle_row_weights(*a.head(), int(token), int(head), _ptr(w), _ptr(o))
    if rc != 0:
        raise OracleError(rc)
    return w, o


def forward_workload(w, nthreads=None, row_ids=None):
    """Oracle on a ``paged_varlen_flash_gb300.workloads.Workload`` (host copies)."""
    kw = dict(causal=w.causal, softcap=w.softcap, window=w.window,
              alibi_slopes=w.alibi_slopes, sinks=w.sinks, nthreads=nthreads,
              k_scale=getattr(w, "k_scale", 1.0), v_scale=getattr(w, "v_scale", 1.0),
              qq_bias=getattr(w, "qq_bias", None), topk_idx=getattr(w, "topk_idx", None),
              topk_len=getattr(w, "topk_len", None))
    if row_ids is None:
        return forward(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                       w.seqused_k, w.scale, **kw)
    return rows(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                w.seqused_k, w.scale, row_ids, **kw)
