"""ctypes binding of libswa.so (include/swa.h), argument marshalling only.

Every compute step runs in the CUDA library; this module checks tensor
types, takes raw device pointers and the current CUDA stream, and calls the
C entry point of the same name.  If the library has not been built the first
call raises: there is no fallback.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswa.so")
# the same library built with SWA_DEBUG_CHECKS (load it first, in its own process)
DEBUG_LIB_PATH = os.path.join(_HERE, "libswa_debug.so")

SWA_OK = 0
SWA_ERR_INVALID_ARG = 1
SWA_ERR_UNSUPPORTED = 2
SWA_ERR_WORKSPACE = 3
SWA_ERR_CUDA = 4
_STATUS = {0: "SWA_OK", 1: "SWA_ERR_INVALID_ARG", 2: "SWA_ERR_UNSUPPORTED",
           3: "SWA_ERR_WORKSPACE", 4: "SWA_ERR_CUDA"}


class SwaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_len", ctypes.c_int32),
                ("num_splits", ctypes.c_int32)]


class SwaPlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("chunk_keys", ctypes.c_int32), ("row_tiles", ctypes.c_int32),
                ("rows_per_tile", ctypes.c_int32), ("grid_ctas", ctypes.c_int32),
                ("merge", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64)]


class SwaDebugOptions(ctypes.Structure):
    """swa_debug_options of include/swa.h (test and sweep controls)."""
    _fields_ = [("force_kernel", ctypes.c_int32), ("pdl", ctypes.c_int32),
                ("wait_limit_cycles", ctypes.c_int64), ("withhold_fill", ctypes.c_int32),
                ("rows_per_item", ctypes.c_int32), ("fail_launch", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


# force_kernel values of swa_debug_options
KERNEL_IDS = {"plan": 0, "simt": 1, "tc": 2, "rows": 3, "pairs": 4}


class SwaError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library(path=LIB_PATH):
    """Load libswa.so and declare the C signatures.  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run sliding_window_speculative_gb300.build.build() "
                          "(nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    lib.swa_verify_attn.argtypes = [vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, vp,
                                    ctypes.POINTER(SwaDims), vp]
    lib.swa_verify_attn.restype = ctypes.c_int
    lib.swa_workspace_bytes.argtypes = [ctypes.POINTER(SwaDims), i32]
    lib.swa_workspace_bytes.restype = sz
    lib.swa_set_workspace.argtypes = [vp, sz]
    lib.swa_set_workspace.restype = ctypes.c_int
    lib.swa_release_workspace.argtypes = []
    lib.swa_release_workspace.restype = ctypes.c_int
    lib.swa_plan.argtypes = [ctypes.POINTER(SwaDims), i32, i32, ctypes.POINTER(SwaPlanInfo)]
    lib.swa_plan.restype = ctypes.c_int
    lib.swa_last_error.argtypes = []
    lib.swa_last_error.restype = ctypes.c_char_p
    lib.swa_read_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.swa_read_device_errors.restype = ctypes.c_int
    lib.swa_read_debug_checks.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.swa_read_debug_checks.restype = ctypes.c_int
    lib.swa_version.argtypes = []
    lib.swa_version.restype = ctypes.c_char_p
    lib.swa_verify_attn_noalloc.argtypes = lib.swa_verify_attn.argtypes
    lib.swa_verify_attn_noalloc.restype = ctypes.c_int
    lib.swa_verify_attn_paged.argtypes = [vp, vp, vp, ctypes.POINTER(SwaPaged), vp, vp, i32,
                                          ctypes.c_float, vp, vp, ctypes.POINTER(SwaDims), vp]
    lib.swa_verify_attn_paged.restype = ctypes.c_int
    lib.swa_append_verify_attn.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(SwaPaged), vp, vp,
                                           i32, ctypes.c_float, vp, vp, ctypes.POINTER(SwaDims),
                                           vp]
    lib.swa_append_verify_attn.restype = ctypes.c_int
    lib.swa_greedy_accept.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
    lib.swa_greedy_accept.restype = ctypes.c_int
    lib.swa_set_debug_options.argtypes = [ctypes.POINTER(SwaDebugOptions)]
    lib.swa_set_debug_options.restype = ctypes.c_int
    lib.swa_get_debug_options.argtypes = [ctypes.POINTER(SwaDebugOptions)]
    lib.swa_get_debug_options.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status):
    if status != SWA_OK:
        raise SwaError(status, swa_last_error())


class SwaPaged(ctypes.Structure):
    """swa_paged of include/swa.h."""
    _fields_ = [("block_table", ctypes.c_void_p), ("max_blocks", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _marshal_paged(q, k_pages, v_pages, block_table, seq_lens, q_pos, window, scale,
                   out=None, lse=None, num_splits=0, stream=None):
    B, q_len, Hq, D = q.shape
    pq = _dev_tensor(q, "q", torch.bfloat16, 4)
    pk = _dev_tensor(k_pages, "k_pages", torch.bfloat16, 4)
    pv = _dev_tensor(v_pages, "v_pages", torch.bfloat16, 4)
    if v_pages.shape != k_pages.shape or k_pages.shape[3] != D:
        raise ValueError("k_pages / v_pages shapes do not match each other or q")
    pt = _dev_tensor(block_table, "block_table", torch.int32, 2)
    if block_table.shape[0] != B:
        raise ValueError("block_table needs one row per sequence")
    ps = _dev_tensor(seq_lens, "seq_lens", torch.int32, 1)
    pp = _dev_tensor(q_pos, "q_pos", torch.int32, 1)
    if out is None:
        out = torch.empty_like(q)
    po = _dev_tensor(out, "out", torch.bfloat16, 4)
    if lse is None:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    pl = _dev_tensor(lse, "lse", torch.float32, 3)
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    max_blocks = block_table.shape[1]
    paged = SwaPaged(pt, max_blocks, page_size, num_pages)
    dims = make_dims(B, q_len, Hq, Hkv, D, max_blocks * page_size, num_splits)
    handle = _stream_handle(stream, q.device)
    args = (pq, pk, pv, ctypes.byref(paged), ps, pp, int(window), float(scale), po, pl,
            ctypes.byref(dims), handle)
    keep = (q, k_pages, v_pages, block_table, seq_lens, q_pos, out, lse, paged, dims)
    return "swa_verify_attn_paged", args, keep, (out, lse)


def swa_verify_attn_paged(q, k_pages, v_pages, block_table, seq_lens, q_pos, window, scale,
                          out=None, lse=None, num_splits=0, stream=None):
    """Windowed verify attention over a paged cache (C entry point
    swa_verify_attn_paged).

    k_pages, v_pages bf16 [num_pages, Hkv, page_size, D]; block_table int32
    [B, max_blocks] (device): block k of sequence b is page
    block_table[b, k].  Everything else as swa_verify_attn.
    """
    return _issue(*_marshal_paged(q, k_pages, v_pages, block_table, seq_lens, q_pos, window,
                                  scale, out, lse, num_splits, stream))


def _issue(entry, args, keep, result):
    _check(getattr(load_library(), entry)(*args))
    return result


def _marshal_append(q, k_new, v_new, k_cache, v_cache, seq_lens, q_pos, window, scale,
                    block_table=None, out=None, lse=None, num_splits=0, stream=None):
    B, q_len, Hq, D = q.shape
    pq = _dev_tensor(q, "q", torch.bfloat16, 4)
    pkn = _dev_tensor(k_new, "k_new", torch.bfloat16, 4)
    pvn = _dev_tensor(v_new, "v_new", torch.bfloat16, 4)
    pk = _dev_tensor(k_cache, "k_cache", torch.bfloat16, 4)
    pv = _dev_tensor(v_cache, "v_cache", torch.bfloat16, 4)
    Hkv = k_cache.shape[1]
    if v_cache.shape != k_cache.shape or k_cache.shape[3] != D:
        raise ValueError("k_cache / v_cache shapes do not match each other or q")
    if k_new.shape != (B, q_len, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [B, q_len, Hkv, D] = %s" % ((B, q_len, Hkv, D),))
    ps = _dev_tensor(seq_lens, "seq_lens", torch.int32, 1)
    pp = _dev_tensor(q_pos, "q_pos", torch.int32, 1)
    if out is None:
        out = torch.empty_like(q)
    po = _dev_tensor(out, "out", torch.bfloat16, 4)
    if lse is None:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    pl = _dev_tensor(lse, "lse", torch.float32, 3)
    paged = None
    if block_table is not None:
        pt = _dev_tensor(block_table, "block_table", torch.int32, 2)
        if block_table.shape[0] != B:
            raise ValueError("block_table needs one row per sequence")
        num_pages, page_size = k_cache.shape[0], k_cache.shape[2]
        paged = SwaPaged(pt, block_table.shape[1], page_size, num_pages)
        max_len = block_table.shape[1] * page_size
    else:
        max_len = k_cache.shape[2]
    dims = make_dims(B, q_len, Hq, Hkv, D, max_len, num_splits)
    handle = _stream_handle(stream, q.device)
    args = (pq, pkn, pvn, pk, pv, ctypes.byref(paged) if paged is not None else None, ps, pp,
            int(window), float(scale), po, pl, ctypes.byref(dims), handle)
    keep = (q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, q_pos, out, lse, paged,
            dims)
    return "swa_append_verify_attn", args, keep, (out, lse)


def swa_append_verify_attn(q, k_new, v_new, k_cache, v_cache, seq_lens, q_pos, window, scale,
                           block_table=None, out=None, lse=None, num_splits=0, stream=None):
    """Fused KV append + windowed verify attention (C entry point
    swa_append_verify_attn): writes k_new / v_new bf16 [B, q_len, Hkv, D]
    into the cache at positions q_pos + i, then attends over the updated
    cache.  Without block_table the caches are [B, Hkv, max_len, D]; with it
    they are page pools [num_pages, Hkv, page_size, D] as in
    swa_verify_attn_paged.  The caches are modified in place.
    """
    return _issue(*_marshal_append(q, k_new, v_new, k_cache, v_cache, seq_lens, q_pos, window,
                                   scale, block_table, out, lse, num_splits, stream))


def make_dims(batch, q_len, num_q_heads, num_kv_heads, head_dim, max_len, num_splits=0):
    return SwaDims(batch, q_len, num_q_heads, num_kv_heads, head_dim, max_len, num_splits)


def dims_of(q, k_cache, num_splits=0):
    B, q_len, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    return make_dims(B, q_len, Hq, Hkv, D, L, num_splits)


def _dev_tensor(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions (got {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _marshal_verify(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out=None, lse=None,
                    num_splits=0, stream=None, want_lse=True, entry="swa_verify_attn"):
    B, q_len, Hq, D = q.shape
    pq = _dev_tensor(q, "q", torch.bfloat16, 4)
    pk = _dev_tensor(k_cache, "k_cache", torch.bfloat16, 4)
    pv = _dev_tensor(v_cache, "v_cache", torch.bfloat16, 4)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError("cache shape does not match q")
    ps = _dev_tensor(seq_lens, "seq_lens", torch.int32, 1)
    pp = _dev_tensor(q_pos, "q_pos", torch.int32, 1)
    if seq_lens.numel() != B or q_pos.numel() != B:
        raise ValueError("seq_lens and q_pos need one entry per sequence")
    if out is None:
        out = torch.empty_like(q)
    po = _dev_tensor(out, "out", torch.bfloat16, 4)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if lse is None and want_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    pl = None
    if lse is not None:
        pl = _dev_tensor(lse, "lse", torch.float32, 3)
        if tuple(lse.shape) != (B, q_len, Hq):
            raise ValueError("lse must be [B, q_len, Hq]")
    dims = dims_of(q, k_cache, num_splits)
    handle = _stream_handle(stream, q.device)
    args = (pq, pk, pv, ps, pp, int(window), float(scale), po, pl, ctypes.byref(dims), handle)
    keep = (q, k_cache, v_cache, seq_lens, q_pos, out, lse, dims)
    return entry, args, keep, (out, lse)


def swa_verify_attn(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out=None, lse=None,
                    num_splits=0, stream=None, want_lse=True):
    """Windowed verify attention through the C entry point swa_verify_attn.

    q bf16 [B, q_len, Hq, D]; k_cache, v_cache bf16 [B, Hkv, L, D];
    seq_lens, q_pos int32 [B] (device).  Returns (out, lse); out/lse are
    allocated if not given (lse only if want_lse).  Enqueued on `stream`
    (default: torch's current stream); does not synchronise.
    """
    return _issue(*_marshal_verify(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse,
                                   num_splits, stream, want_lse))


def _marshal_noalloc(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse=None,
                     num_splits=0, stream=None):
    if out is None:
        raise ValueError("swa_verify_attn_noalloc writes into a caller-given out tensor")
    return _marshal_verify(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse,
                           num_splits, stream, want_lse=False, entry="swa_verify_attn_noalloc")


def swa_verify_attn_noalloc(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out, lse=None,
                            num_splits=0, stream=None):
    """The allocation-free C entry point swa_verify_attn_noalloc: same
    arguments as swa_verify_attn, but `out` (and `lse`, if wanted) must be
    given, and split partials use the library's fixed 16 MiB device scratch
    instead of a cudaMalloc'd workspace.  For callers that may not allocate
    device memory while serving (a pre-reserved memory pool, a framework that
    owns every allocation, a path that cannot take cudaMalloc's device
    synchronisation).  Overlapping calls on one device share the scratch and
    race; make the first call on a device outside stream capture."""
    return _issue(*_marshal_noalloc(q, k_cache, v_cache, seq_lens, q_pos, window, scale, out,
                                    lse, num_splits, stream))


class PreparedCall:
    """One attention call validated and marshalled once (see prepare()).

    Calling the object re-issues the same C call with the same pointers,
    shapes, window, scale and stream; the tensors' contents may change
    between calls (a serving loop writes the next step's rows into the same
    buffers).  Returns the (out, lse) tensors the call writes.  The object
    keeps every tensor it points at alive."""

    def __init__(self, entry, args, keep, result):
        self._fn = getattr(load_library(), entry)
        self.entry = entry
        self._args = args
        self._keep = keep
        self.result = result

    def __call__(self):
        st = self._fn(*self._args)
        if st != SWA_OK:
            _check(st)
        return self.result


_MARSHAL = {"swa_verify_attn": _marshal_verify, "swa_verify_attn_noalloc": _marshal_noalloc,
            "swa_verify_attn_paged": _marshal_paged, "swa_append_verify_attn": _marshal_append}


def prepare(fn, *args, **kwargs):
    """Validate and marshal a call of swa_verify_attn, swa_verify_attn_noalloc,
    swa_verify_attn_paged or swa_append_verify_attn once, with the same
    arguments the function takes, and return a PreparedCall that issues it.

    The per-call host cost is then one C call: no tensor checks, no struct
    building, no stream lookup (the stream is the one given, or torch's
    current stream at prepare time).  Outputs are allocated here if not
    given."""
    name = fn if isinstance(fn, str) else fn.__name__
    if name not in _MARSHAL:
        raise ValueError(f"cannot prepare {name}; one of {sorted(_MARSHAL)}")
    return PreparedCall(*_MARSHAL[name](*args, **kwargs))


def swa_greedy_accept(logits, draft=None, keep_ids=None, argmax=None, accepted=None,
                      stream=None):
    """Greedy verification through the C entry point swa_greedy_accept.

    logits bf16 [B, q_len, V]; draft int32 [B, q_len - 1] (None when
    q_len == 1); keep_ids int32 [V] or None.  Returns (argmax int32
    [B, q_len], accepted int32 [B]), allocated if not given.  Enqueued on
    `stream` (default: torch's current stream); does not synchronise.
    """
    lib = load_library()
    pl = _dev_tensor(logits, "logits", torch.bfloat16, 3)
    B, q_len, V = logits.shape
    pd = None
    if q_len > 1 or draft is not None:
        pd = _dev_tensor(draft, "draft", torch.int32, 2)
        if tuple(draft.shape) != (B, q_len - 1):
            raise ValueError("draft must be [B, q_len - 1]")
    pk = None
    if keep_ids is not None:
        pk = _dev_tensor(keep_ids, "keep_ids", torch.int32, 1)
        if keep_ids.numel() != V:
            raise ValueError("keep_ids needs one token id per logit column")
    if argmax is None:
        argmax = torch.empty((B, q_len), dtype=torch.int32, device=logits.device)
    if accepted is None:
        accepted = torch.empty((B,), dtype=torch.int32, device=logits.device)
    pa = _dev_tensor(argmax, "argmax", torch.int32, 2)
    pc = _dev_tensor(accepted, "accepted", torch.int32, 1)
    if tuple(argmax.shape) != (B, q_len) or accepted.numel() != B:
        raise ValueError("argmax must be [B, q_len] and accepted [B]")
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(lib.swa_greedy_accept(pl, pk, pd, pa, pc, B, q_len, V, handle))
    return argmax, accepted


def swa_workspace_bytes(dims, window):
    return load_library().swa_workspace_bytes(ctypes.byref(dims), int(window))


def swa_set_workspace(buffer=None):
    """Use a caller-owned CUDA tensor as the current device's workspace
    (None returns to the library-owned buffer)."""
    lib = load_library()
    if buffer is None:
        _check(lib.swa_set_workspace(None, 0))
    else:
        _check(lib.swa_set_workspace(buffer.data_ptr(), buffer.numel() * buffer.element_size()))


def swa_release_workspace():
    _check(load_library().swa_release_workspace())


def swa_plan(dims, window, num_sms):
    info = SwaPlanInfo()
    _check(load_library().swa_plan(ctypes.byref(dims), int(window), int(num_sms),
                                   ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in SwaPlanInfo._fields_}


def swa_last_error():
    return load_library().swa_last_error().decode()


def swa_read_device_errors():
    flags = ctypes.c_uint32(0)
    _check(load_library().swa_read_device_errors(ctypes.byref(flags)))
    return flags.value


def swa_read_debug_checks():
    """Out-of-range index attempts counted since the last read (C entry point
    swa_read_debug_checks; needs the SWA_DEBUG_CHECKS build, else SwaError
    with SWA_ERR_UNSUPPORTED).  Synchronises the device."""
    count = ctypes.c_uint32(0)
    _check(load_library().swa_read_debug_checks(ctypes.byref(count)))
    return count.value


def swa_version():
    return load_library().swa_version().decode()


def swa_set_debug_options(force_kernel=0, pdl=1, wait_limit_cycles=0, withhold_fill=-1,
                          rows_per_item=0, fail_launch=0):
    """Test and sweep controls of the C entry point swa_set_debug_options
    (not for serving).  force_kernel: 0 or "plan", 1 or "simt", 2 or "tc",
    3 or "rows", 4 or "pairs"; pdl 1/0; wait_limit_cycles 0 (default ~2e9) or the bounded
    waits' limit; withhold_fill -1 or the fill the first CTA never copies;
    rows_per_item 0 (the plan's) or packed rows per tensor-core work item;
    fail_launch 0 or n: the n-th library launch from now on is not made and
    its call fails (then back to 0)."""
    fk = KERNEL_IDS[force_kernel] if isinstance(force_kernel, str) else int(force_kernel)
    opt = SwaDebugOptions(fk, int(pdl), int(wait_limit_cycles), int(withhold_fill),
                          int(rows_per_item), int(fail_launch), 0)
    _check(load_library().swa_set_debug_options(ctypes.byref(opt)))


def swa_get_debug_options():
    opt = SwaDebugOptions()
    _check(load_library().swa_get_debug_options(ctypes.byref(opt)))
    return {f: getattr(opt, f) for f, _ in SwaDebugOptions._fields_}
