"""ctypes binding of ``include/ua.h`` (argument marshalling only).

Every function here forwards to the C ABI of ``libua.so``; all arithmetic runs
in that library's CUDA kernels.  Tensors are torch tensors (device memory for
``ua_forward``, host memory for ``ua_forward_host``); streams are torch CUDA
streams or raw ``cudaStream_t`` integers.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libua.so")

UA_OK = 0
UA_FLAG_CAUSAL = 1 << 0
UA_FLAG_SOFTCAP = 1 << 1
UA_FLAG_ALIBI = 1 << 2
UA_FLAG_WINDOW = 1 << 3
UA_FLAG_SINKS = 1 << 4
UA_FLAG_QQ_BIAS = 1 << 5
UA_PARTIALS_F32 = 0
UA_PARTIALS_BF16 = 1

UA_DEVERR_CONTEXT = 1 << 0
UA_DEVERR_BLOCK_ID = 1 << 1
UA_DEVERR_CU_SEQLENS = 1 << 2
UA_DEVERR_BOUNDS = 1 << 3
UA_DEVERR_TIMEOUT = 1 << 4

UA_DTYPE_BF16 = 0
UA_DTYPE_FP8_E4M3 = 1

UA_PATH_AUTO = 0
UA_PATH_SPLIT_KV = 1
UA_PATH_TENSOR_CORE = 2
UA_PATH_DECODE_TC = 3

_lib = None


class UAError(RuntimeError):
    def __init__(self, status, what=""):
        msg = "%s: %s" % (what or "ua", ua_status_string(status))
        if status == 3 and _lib is not None:
            msg += " (%s)" % _lib.ua_last_cuda_error().decode()
        super().__init__(msg)
        self.status = status


class ProblemDesc(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_size", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64),
        ("max_num_seqs", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_total_q", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("window", ctypes.c_int32),
        ("path", ctypes.c_uint32),
        ("kv_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("split_partials", ctypes.c_int32),
    ]


def lib_path():
    return _LIB_PATH


def load_library():
    """Load ``libua.so``; raise if it has not been built (no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            "libua.so is not built (%s); run `python -m paged_varlen_flash_gb300.build`"
            % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    lib.ua_problem_create.argtypes = [ctypes.POINTER(ProblemDesc), ctypes.POINTER(vp)]
    lib.ua_problem_create.restype = ctypes.c_int
    fwd = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, u32, vp, vp, vp, vp]
    lib.ua_forward.argtypes = fwd
    lib.ua_forward.restype = ctypes.c_int
    lib.ua_forward_host.argtypes = fwd
    lib.ua_forward_host.restype = ctypes.c_int
    lib.ua_check_device_error.argtypes = [vp, vp, ctypes.POINTER(i32)]
    lib.ua_check_device_error.restype = ctypes.c_int
    lib.ua_last_launch_count.argtypes = [vp]
    lib.ua_last_launch_count.restype = i32
    lib.ua_last_path.argtypes = [vp]
    lib.ua_last_path.restype = ctypes.c_char_p
    lib.ua_forward_topk.argtypes = [vp] * 7 + [i32, ctypes.c_int64, i32, i32, vp, vp, i32,
                                               ctypes.c_uint32, vp, vp, vp, vp]
    lib.ua_forward_topk.restype = ctypes.c_int
    lib.ua_set_qq_bias.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int64]
    lib.ua_set_qq_bias.restype = ctypes.c_int
    lib.ua_debug_stall_data_waits.argtypes = [vp, i32, i64]
    lib.ua_debug_stall_data_waits.restype = ctypes.c_int
    lib.ua_set_profile_events.argtypes = [vp, vp, vp]
    lib.ua_set_profile_events.restype = ctypes.c_int
    lib.ua_destroy.argtypes = [vp]
    lib.ua_destroy.restype = None
    lib.ua_status_string.argtypes = [ctypes.c_int]
    lib.ua_status_string.restype = ctypes.c_char_p
    lib.ua_last_cuda_error.argtypes = []
    lib.ua_last_cuda_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def ua_status_string(status):
    return load_library().ua_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def flags_of(causal=True, softcap=0.0, alibi=False, window=0, sinks=False, qq_bias=False):
    f = 0
    if causal:
        f |= UA_FLAG_CAUSAL
    if softcap:
        f |= UA_FLAG_SOFTCAP
    if alibi:
        f |= UA_FLAG_ALIBI
    if window:
        f |= UA_FLAG_WINDOW
    if sinks:
        f |= UA_FLAG_SINKS
    if qq_bias:
        f |= UA_FLAG_QQ_BIAS
    return f


def ua_problem_create(num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                      max_num_seqs, max_blocks_per_seq, max_total_q, flags, scale,
                      softcap=0.0, window=0, path=UA_PATH_AUTO, kv_dtype=UA_DTYPE_BF16,
                      k_scale=1.0, v_scale=1.0, split_partials=UA_PARTIALS_F32):
    """Returns an opaque problem handle (int); raises UAError on failure."""
    lib = load_library()
    d = ProblemDesc(num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                    max_num_seqs, max_blocks_per_seq, max_total_q, UA_DTYPE_BF16, flags,
                    scale, softcap, window, path, kv_dtype, k_scale, v_scale, split_partials)
    h = ctypes.c_void_p()
    st = lib.ua_problem_create(ctypes.byref(d), ctypes.byref(h))
    if st != UA_OK:
        raise UAError(st, "ua_problem_create")
    return h.value


def ua_forward(problem, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
               num_seqs, total_q, max_seqlen_q, max_seqlen_k, flags, sinks, alibi_slopes,
               out, stream=None):
    """Enqueue a forward pass; all tensors are device tensors.  Returns the
    status code (0 = ok) without raising, so callers can test error paths."""
    return load_library().ua_forward(
        problem, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(cu_seqlens_q), _ptr(seqused_k), num_seqs, total_q, max_seqlen_q,
        max_seqlen_k, flags, _ptr(sinks), _ptr(alibi_slopes), _ptr(out), _stream(stream))


def ua_forward_topk(problem, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                    num_seqs, total_q, max_seqlen_q, max_seqlen_k, topk_idx, topk_len,
                    topk_stride, flags, sinks, alibi_slopes, out, stream=None):
    """Enqueue a sparse top-k forward (device tensors; topk_idx int32
    [total_q, topk_stride], topk_len int32 [total_q]).  Returns the status."""
    return load_library().ua_forward_topk(
        problem, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(cu_seqlens_q), _ptr(seqused_k), num_seqs, total_q, max_seqlen_q,
        max_seqlen_k, _ptr(topk_idx), _ptr(topk_len), topk_stride, flags, _ptr(sinks),
        _ptr(alibi_slopes), _ptr(out), _stream(stream))


def ua_forward_host(problem, q_host, k_cache, v_cache, block_table_host, cu_seqlens_q_host,
                    seqused_k_host, num_seqs, total_q, max_seqlen_q, max_seqlen_k, flags,
                    sinks_host, alibi_host, out_host, stream=None):
    """Forward with host-resident per-step inputs and output (caches on device)."""
    return load_library().ua_forward_host(
        problem, _ptr(q_host), _ptr(k_cache), _ptr(v_cache), _ptr(block_table_host),
        _ptr(cu_seqlens_q_host), _ptr(seqused_k_host), num_seqs, total_q, max_seqlen_q,
        max_seqlen_k, flags, _ptr(sinks_host), _ptr(alibi_host), _ptr(out_host),
        _stream(stream))


def ua_forward_noalloc(desc, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                       num_seqs, total_q, max_seqlen_q, max_seqlen_k, flags, sinks,
                       alibi_slopes, out, device_error=None, stream=None):
    """The allocation-free forward (``ProblemDesc`` instead of a problem
    handle; partials in the library's static device scratch).  Returns the
    status code without raising."""
    lib = load_library()
    fn = lib.ua_forward_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(ProblemDesc), vp, vp, vp, vp, vp, vp, ctypes.c_int32,
                   ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32, vp, vp,
                   vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
              _ptr(cu_seqlens_q), _ptr(seqused_k), num_seqs, total_q, max_seqlen_q,
              max_seqlen_k, flags, _ptr(sinks), _ptr(alibi_slopes), _ptr(out),
              _ptr(device_error), _stream(stream))


def ua_set_qq_bias(problem, bias, n, row_stride):
    """Bind the query-query bias matrix (device fp32, element (a, c) at
    a * row_stride + c) to a problem; ``bias=None`` clears it.  Returns the
    status code without raising."""
    return load_library().ua_set_qq_bias(problem, _ptr(bias), n, row_stride)


def ua_debug_stall_data_waits(problem, enable, limit_ns=2_000_000):
    """Testing hook: make the next forward calls' first K/V data wait run out
    after ``limit_ns`` (see include/ua.h).  Returns the status code."""
    return load_library().ua_debug_stall_data_waits(problem, int(enable), int(limit_ns))


def ua_check_device_error(problem, stream=None):
    """Synchronise the stream and return (and clear) the device error word."""
    code = ctypes.c_int32(0)
    st = load_library().ua_check_device_error(problem, _stream(stream), ctypes.byref(code))
    if st not in (UA_OK, 5):
        raise UAError(st, "ua_check_device_error")
    return code.value


def ua_destroy(problem):
    if problem:
        load_library().ua_destroy(problem)


class Problem:
    """Owning wrapper around a ``ua_problem`` handle."""

    def __init__(self, num_q_heads, num_kv_heads, head_size, block_size, num_blocks,
                 max_num_seqs, max_blocks_per_seq, max_total_q, flags, scale, softcap=0.0,
                 window=0, path=UA_PATH_AUTO, kv_dtype=UA_DTYPE_BF16, k_scale=1.0, v_scale=1.0,
                 split_partials=UA_PARTIALS_F32):
        self.handle = ua_problem_create(num_q_heads, num_kv_heads, head_size, block_size,
                                        num_blocks, max_num_seqs, max_blocks_per_seq,
                                        max_total_q, flags, scale, softcap, window, path,
                                        kv_dtype, k_scale, v_scale, split_partials)
        self.flags = flags
        self.head_size = head_size
        self.num_q_heads = num_q_heads

    @classmethod
    def for_workload(cls, w, max_total_q=None, max_num_seqs=None, extra_flags=0,
                     path=UA_PATH_AUTO, split_partials=UA_PARTIALS_F32):
        flags = flags_of(w.causal, w.softcap, w.alibi_slopes is not None, w.window,
                         w.sinks is not None, getattr(w, "qq_bias", None) is not None) | extra_flags
        fp8 = getattr(w, "kv_fp8", False)
        return cls(w.hq, w.hk, w.d, w.b, w.num_blocks, max_num_seqs or max(1, w.num_seqs),
                   w.max_blocks_per_seq, max_total_q or max(1, w.total_q), flags, w.scale,
                   w.softcap, w.window, path, UA_DTYPE_FP8_E4M3 if fp8 else UA_DTYPE_BF16,
                   getattr(w, "k_scale", 1.0), getattr(w, "v_scale", 1.0), split_partials)

    def forward(self, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k, num_seqs,
                total_q, max_seqlen_q, max_seqlen_k, flags, sinks=None, alibi_slopes=None,
                out=None, stream=None):
        if out is None:
            import torch
            out = torch.empty_like(q)
        st = ua_forward(self.handle, q, k_cache, v_cache, block_table, cu_seqlens_q,
                        seqused_k, num_seqs, total_q, max_seqlen_q, max_seqlen_k, flags,
                        sinks, alibi_slopes, out, stream)
        if st != UA_OK:
            raise UAError(st, "ua_forward")
        return out

    def forward_topk(self, q, k_cache, v_cache, block_table, cu_seqlens_q, seqused_k,
                     num_seqs, total_q, max_seqlen_q, max_seqlen_k, topk_idx, topk_len, flags,
                     sinks=None, alibi_slopes=None, out=None, stream=None):
        if out is None:
            import torch
            out = torch.empty_like(q)
        if topk_idx.dim() != 2 or topk_idx.stride(1) != 1:
            raise ValueError("topk_idx must be [total_q, K] with unit inner stride")
        st = ua_forward_topk(self.handle, q, k_cache, v_cache, block_table, cu_seqlens_q,
                             seqused_k, num_seqs, total_q, max_seqlen_q, max_seqlen_k, topk_idx,
                             topk_len, topk_idx.stride(0), flags, sinks, alibi_slopes, out,
                             stream)
        if st != UA_OK:
            raise UAError(st, "ua_forward_topk")
        return out

    def forward_workload(self, w, out=None, stream=None):
        """Forward on a device-resident ``workloads.Workload`` (through
        ``ua_forward_topk`` when it carries top-k lists)."""
        qq = getattr(w, "qq_bias", None)
        flags = flags_of(w.causal, w.softcap, w.alibi_slopes is not None, w.window,
                         w.sinks is not None, qq is not None)
        if qq is not None:
            self.set_qq_bias(qq)
        if getattr(w, "topk_idx", None) is not None:
            return self.forward_topk(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                                     w.seqused_k, w.num_seqs, w.total_q, w.max_seqlen_q,
                                     w.max_seqlen_k, w.topk_idx, w.topk_len, flags, w.sinks,
                                     w.alibi_slopes, out, stream)
        return self.forward(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                            w.seqused_k, w.num_seqs, w.total_q, w.max_seqlen_q,
                            w.max_seqlen_k, flags, w.sinks, w.alibi_slopes, out, stream)

    def set_qq_bias(self, bias):
        """Bind a device fp32 matrix [n, >= n] (unit inner stride) as the
        query-query bias of later calls with UA_FLAG_QQ_BIAS; None clears it.
        The problem keeps a reference so the memory outlives its use."""
        if bias is None:
            st = ua_set_qq_bias(self.handle, None, 0, 0)
        else:
            if bias.dim() != 2 or bias.stride(1) != 1 or bias.shape[1] < bias.shape[0]:
                raise ValueError("qq bias must be [n, >= n] with unit inner stride")
            st = ua_set_qq_bias(self.handle, bias, bias.shape[0], bias.stride(0))
        if st != UA_OK:
            raise UAError(st, "ua_set_qq_bias")
        self._qq_bias = bias

    def check_device_error(self, stream=None):
        return ua_check_device_error(self.handle, stream)

    def last_launch_count(self):
        return load_library().ua_last_launch_count(self.handle)

    def set_profile_events(self, ev_begin=None, ev_end=None):
        """Record torch.cuda.Event pairs around the dominant kernel of later
        forward calls (None, None switches the hook off)."""
        b = ev_begin.cuda_event if ev_begin is not None else None
        e = ev_end.cuda_event if ev_end is not None else None
        st = load_library().ua_set_profile_events(self.handle, b, e)
        if st != UA_OK:
            raise UAError(st, "ua_set_profile_events")

    def last_path(self):
        return load_library().ua_last_path(self.handle).decode()

    def close(self):
        if self.handle:
            ua_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
