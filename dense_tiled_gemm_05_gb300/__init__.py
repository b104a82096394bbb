"""Python binding of the GB300 blocked-GEMM library (``include/gemm.h``).

The binding only marshals arguments: it reads shapes, strides, data pointers
and the current CUDA stream from torch tensors and calls the C ABI through
ctypes. Every step of the product runs in the library's own CUDA kernels; if
the compiled library is missing, importing the binding's entry points raises
instead of falling back to anything else.

    import dense_tiled_gemm_05_gb300 as g
    c = g.matmul(a, b)                       # a: M x K, b: K x N, CUDA tensors
    c = g.matmul(a32, b32, precision="tf32") # fp32 inputs on the tf32 tensor cores

Layouts follow the tensors' strides: a row-major view has stride (ld, 1), a
column-major view stride (1, ld) (e.g. ``b_storage.t()`` for a B stored as
[N, K]). The output is row-major.
"""
import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libgemm_gb300.so")

# enums of include/gemm.h
F32, F16, BF16 = 0, 1, 2
PREC = {"default": 0, "tf32": 1, "exact": 2, "f16acc": 3}
ROW, COL = 0, 1
STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED",
          3: "GEMM_ERR_ALIGNMENT", 4: "GEMM_ERR_NO_MEMORY", 5: "GEMM_ERR_CUDA",
          6: "GEMM_ERR_TIMEOUT", 7: "GEMM_ERR_DEVICE"}
OPTIONS = {"wait_timeout_us": 0, "force_path": 1, "group_m": 2, "max_ctas": 3,
           "fault_stall_producer": 4, "force_staging": 5, "cta_pair": 6,
           "block_n": 7, "exact_chunk": 8, "stream_k": 9, "host_panel": 10, "acc_chunk": 11, "stage_k": 12,
           "tile_rows": 13, "tf32_transpose": 14}
PATHS = {0: "none", 1: "zero_fill", 2: "tcgen05", 3: "fma", 4: "tcgen05_3xtf32",
         5: "tcgen05_f16acc"}
_DT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
_DT_NAMES = {"f32": F32, "f16": F16, "bf16": BF16}
_TORCH_OF = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}

# Every symbol include/gemm.h declares.
EXPORTS = ("gemm_create", "gemm_destroy", "gemm_run", "gemm_run_ex", "gemm_get_status",
           "gemm_strerror", "gemm_set_option", "gemm_get_launch_count", "gemm_plan",
           "gemm_version", "gemm_run_noalloc", "gemm_schedule_segments", "gemm_run_host",
           "gemm_run_strided", "gemm_plan_strided", "gemm_tune", "gemm_tune_clear",
           "gemm_softmax_rows", "gemm_set_kernel_events")


class GemmError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        self.status = STATUS.get(code, str(code))
        super().__init__("%s%s (%s)" % (what + ": " if what else "", self.status, _strerror(code)))


class TuneResult(ctypes.Structure):
    _fields_ = [("cta_pair", ctypes.c_int32), ("block_n", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("stage_k", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("tile_rows", ctypes.c_int32),
                ("candidates", ctypes.c_int32),
                ("best_us", ctypes.c_float), ("default_us", ctypes.c_float)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class StridedInfo(ctypes.Structure):
    _fields_ = [("a_gathered", ctypes.c_int32), ("b_gathered", ctypes.c_int32),
                ("c_mode", ctypes.c_int32), ("buffer_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("grid_m", ctypes.c_int64), ("grid_n", ctypes.c_int64),
                ("k_iters", ctypes.c_int64), ("stages", ctypes.c_int32), ("stage_a", ctypes.c_int32),
                ("stage_b", ctypes.c_int32), ("a_mn_major", ctypes.c_int32),
                ("b_mn_major", ctypes.c_int32), ("tma_store", ctypes.c_int32),
                ("ctas", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("cta_pair", ctypes.c_int32), ("split_tiles", ctypes.c_int32)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["path"] = PATHS.get(d["path"], d["path"])
        return d


_lib = None
_lib_lock = threading.Lock()


def lib():
    """The loaded C library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        "libgemm_gb300.so is not built; run "
                        "`python -c 'import __graft_entry__ as g; g.build()'` "
                        "(or python dense_tiled_gemm_05_gb300/build.py)")
                L = ctypes.CDLL(LIB_PATH)
                i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
                run_args = [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32]
                L.gemm_create.argtypes = [ctypes.POINTER(vp), i32]
                L.gemm_create.restype = i32
                L.gemm_destroy.argtypes = [vp]
                L.gemm_destroy.restype = None
                L.gemm_run.argtypes = run_args
                L.gemm_run.restype = i32
                L.gemm_run_ex.argtypes = run_args + [i32, i32, vp]
                L.gemm_run_ex.restype = i32
                L.gemm_run_host.argtypes = run_args + [i32, i32, vp]
                L.gemm_run_host.restype = i32
                strided = [vp, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, i32,
                           i32, i32]
                L.gemm_run_strided.argtypes = strided + [vp]
                L.gemm_run_strided.restype = i32
                L.gemm_plan_strided.argtypes = strided + [i32, ctypes.POINTER(PlanInfo),
                                                          ctypes.POINTER(StridedInfo)]
                L.gemm_plan_strided.restype = i32
                L.gemm_tune.argtypes = run_args + [i32, i32, vp, i32, ctypes.POINTER(TuneResult)]
                L.gemm_tune.restype = i32
                L.gemm_softmax_rows.argtypes = [vp, i64, i64, vp, i64, vp, i64, i32, i32, vp]
                L.gemm_softmax_rows.restype = i32
                L.gemm_tune_clear.argtypes = [vp]
                L.gemm_tune_clear.restype = i32
                L.gemm_get_status.argtypes = [vp, vp]
                L.gemm_get_status.restype = i32
                L.gemm_strerror.argtypes = [i32]
                L.gemm_strerror.restype = ctypes.c_char_p
                L.gemm_set_option.argtypes = [vp, i32, i64]
                L.gemm_set_option.restype = i32
                L.gemm_get_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
                L.gemm_get_launch_count.restype = i32
                L.gemm_set_kernel_events.argtypes = [vp, vp, vp]
                L.gemm_set_kernel_events.restype = i32
                L.gemm_plan.argtypes = run_args + [i32, i32, ctypes.c_int32,
                                                   ctypes.POINTER(PlanInfo)]
                L.gemm_plan.restype = i32
                L.gemm_run_noalloc.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32,
                                               i32, i32, i32, i32, vp, vp]
                L.gemm_run_noalloc.restype = i32
                L.gemm_schedule_segments.argtypes = [i32, i32, i32, i32, i32,
                                                     ctypes.POINTER(ctypes.c_int32), vp, i32]
                L.gemm_schedule_segments.restype = i32
                L.gemm_version.argtypes = []
                L.gemm_version.restype = ctypes.c_char_p
                _lib = L
    return _lib


def _strerror(code):
    try:
        return lib().gemm_strerror(code).decode()
    except RuntimeError:
        return "library not loaded"


def _check(code, what=""):
    if code != 0:
        raise GemmError(code, what)


def operand_layout(x):
    """(layout, ld) of a 2-D view: ROW for stride (ld, 1), COL for stride (1, ld)."""
    if x.dim() != 2:
        raise ValueError("operands must be 2-D")
    r, c = x.shape
    s0, s1 = x.stride()
    if s1 == 1 and (s0 >= max(c, 1) or r <= 1):
        return ROW, max(s0, c, 1)
    if s0 == 1 and (s1 >= max(r, 1) or c <= 1):
        return COL, max(s1, r, 1)
    raise ValueError("operand must be row- or column-major, got stride %s" % (x.stride(),))


def _dtype_code(d):
    if isinstance(d, str):
        return _DT_NAMES[d]
    if d in _DT:
        return _DT[d]
    raise TypeError("unsupported dtype %s" % d)


class Gemm:
    """A library handle bound to one CUDA device."""

    def __init__(self, device=None):
        if device is None:
            device = torch.cuda.current_device()
        self.device = int(device)
        h = ctypes.c_void_p()
        _check(lib().gemm_create(ctypes.byref(h), self.device), "gemm_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().gemm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def set_option(self, name, value):
        _check(lib().gemm_set_option(self._h, OPTIONS[name], int(value)), "gemm_set_option")

    def launch_count(self):
        n = ctypes.c_uint64()
        _check(lib().gemm_get_launch_count(self._h, ctypes.byref(n)))
        return n.value

    def set_kernel_events(self, start=None, end=None):
        """Record two torch.cuda.Event objects around the main GEMM kernel of every later
        product on this handle (after any staging copies); no arguments turn it off. The
        events must have been recorded once, so that their CUDA events exist."""
        if start is None or end is None:
            _check(lib().gemm_set_kernel_events(self._h, None, None), "gemm_set_kernel_events")
            self._kernel_events = None
            return
        self._kernel_events = (start, end)  # kept alive while the hook is set
        _check(lib().gemm_set_kernel_events(self._h, ctypes.c_void_p(start.cuda_event),
                                            ctypes.c_void_p(end.cuda_event)),
               "gemm_set_kernel_events")

    def status(self, stream=None):
        """Synchronise the stream and return the device status code (0 = OK), cleared."""
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        return lib().gemm_get_status(self._h, ctypes.c_void_p(s.cuda_stream))

    def run_raw(self, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision=0,
                a_layout=ROW, b_layout=COL, stream=0):
        """Direct C-ABI call with integer pointers; returns the status code."""
        return lib().gemm_run_ex(self._h, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype,
                                 precision, a_layout, b_layout, ctypes.c_void_p(stream))

    def matmul(self, a, b, out=None, out_dtype=None, precision="default", stream=None):
        """C = a @ b on the GPU; a is M x K, b is K x N, out M x N: any 2-D views (row- or
        column-major views go through gemm_run_ex, others through gemm_run_strided)."""
        if a.dtype != b.dtype:
            raise TypeError("a and b must share a dtype")
        if not (a.is_cuda and b.is_cuda):
            raise ValueError("operands must be CUDA tensors (see matmul_host for host buffers)")
        if a.dim() != 2 or b.dim() != 2:
            raise ValueError("operands must be 2-D")
        M, K = a.shape
        K2, N = b.shape
        if K != K2:
            raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
        in_dt = _dtype_code(a.dtype)
        if out is None:
            od = _TORCH_OF[_dtype_code(out_dtype)] if out_dtype is not None else a.dtype
            out = torch.empty((M, N), dtype=od, device=a.device)
        if out.dim() != 2 or out.shape != (M, N):
            raise ValueError("out must be an M x N tensor")
        s = torch.cuda.current_stream(a.device) if stream is None else stream
        ptr = lambda t: ctypes.c_void_p(t.data_ptr())
        try:
            al, lda = operand_layout(a)
            bl, ldb = operand_layout(b)
            row_c = (N <= 1 or out.stride(1) == 1) and (M <= 1 or out.stride(0) >= N)
        except ValueError:
            row_c = False
        if row_c:
            ldc = max(out.stride(0) if M > 1 else N, N, 1)
            code = lib().gemm_run_ex(self._h, M, N, K, ptr(a), lda, ptr(b), ldb, ptr(out), ldc,
                                     in_dt, _dtype_code(out.dtype), PREC[precision], al, bl,
                                     ctypes.c_void_p(s.cuda_stream))
            _check(code, "gemm_run_ex")
        else:
            code = lib().gemm_run_strided(self._h, M, N, K, ptr(a), a.stride(0), a.stride(1),
                                          ptr(b), b.stride(0), b.stride(1), ptr(out),
                                          out.stride(0), out.stride(1), in_dt,
                                          _dtype_code(out.dtype), PREC[precision],
                                          ctypes.c_void_p(s.cuda_stream))
            _check(code, "gemm_run_strided")
        return out

    def tune(self, a, b, out=None, out_dtype=None, precision="default", iters=5, stream=None):
        """Time the tile-shape configurations for this problem (row- or column-major CUDA
        views) and keep the fastest for its signature on this handle; returns the choice
        as a dict (see gemm_tune). C is written."""
        M, K = a.shape
        N = b.shape[1]
        if out is None:
            od = _TORCH_OF[_dtype_code(out_dtype)] if out_dtype is not None else a.dtype
            out = torch.empty((M, N), dtype=od, device=a.device)
        al, lda = operand_layout(a)
        bl, ldb = operand_layout(b)
        s = torch.cuda.current_stream(a.device) if stream is None else stream
        r = TuneResult()
        code = lib().gemm_tune(self._h, M, N, K, ctypes.c_void_p(a.data_ptr()), lda,
                               ctypes.c_void_p(b.data_ptr()), ldb, ctypes.c_void_p(out.data_ptr()),
                               max(out.stride(0), N, 1), _dtype_code(a.dtype),
                               _dtype_code(out.dtype), PREC[precision], al, bl,
                               ctypes.c_void_p(s.cuda_stream), int(iters), ctypes.byref(r))
        _check(code, "gemm_tune")
        return r.as_dict()

    def softmax_rows(self, x, out=None, out_dtype=None, stream=None):
        """Row softmax of a CUDA matrix with unit column stride (Lesson 4, homework 4):
        out[i] = exp(x[i] - max(x[i])) / sum(exp(x[i] - max(x[i]))). ``out=x`` runs in
        place."""
        if not x.is_cuda or x.dim() != 2:
            raise ValueError("x must be a 2-D CUDA tensor")
        M, N = x.shape
        if N > 1 and x.stride(1) != 1:
            raise ValueError("rows of x must be contiguous")
        if out is None:
            od = _TORCH_OF[_dtype_code(out_dtype)] if out_dtype is not None else x.dtype
            out = torch.empty((M, N), dtype=od, device=x.device)
        if out.shape != (M, N) or (N > 1 and out.stride(1) != 1):
            raise ValueError("out must be an M x N tensor with contiguous rows")
        s = torch.cuda.current_stream(x.device) if stream is None else stream
        code = lib().gemm_softmax_rows(self._h, M, N, ctypes.c_void_p(x.data_ptr()),
                                       max(x.stride(0) if M > 1 else N, N, 1),
                                       ctypes.c_void_p(out.data_ptr()),
                                       max(out.stride(0) if M > 1 else N, N, 1),
                                       _dtype_code(x.dtype), _dtype_code(out.dtype),
                                       ctypes.c_void_p(s.cuda_stream))
        _check(code, "gemm_softmax_rows")
        return out

    def tune_clear(self):
        _check(lib().gemm_tune_clear(self._h), "gemm_tune_clear")

    def matmul_host(self, a, b, out=None, out_dtype=None, precision="default", stream=None):
        """C = a @ b for HOST tensors through gemm_run_host: the library copies A and B to the
        GPU and C back, overlapping the copies of one row panel with the product of another.

        Pinned host tensors (``pin_memory=True``) give asynchronous copies; the call returns
        once the work is enqueued on the stream, so synchronise before reading ``out``.
        """
        if a.is_cuda or b.is_cuda:
            raise ValueError("matmul_host takes host tensors")
        if a.dtype != b.dtype:
            raise TypeError("a and b must share a dtype")
        M, K = a.shape
        K2, N = b.shape
        if K != K2:
            raise ValueError("inner dimensions differ: %d vs %d" % (K, K2))
        if out is None:
            od = _TORCH_OF[_dtype_code(out_dtype)] if out_dtype is not None else a.dtype
            out = torch.empty((M, N), dtype=od, pin_memory=True)
        if out.is_cuda or out.dim() != 2 or out.shape != (M, N) or (N > 1 and out.stride(1) != 1):
            raise ValueError("out must be a row-major M x N host tensor")
        al, lda = operand_layout(a)
        bl, ldb = operand_layout(b)
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        code = lib().gemm_run_host(self._h, M, N, K, ctypes.c_void_p(a.data_ptr()), lda,
                                   ctypes.c_void_p(b.data_ptr()), ldb,
                                   ctypes.c_void_p(out.data_ptr()), max(out.stride(0), N, 1),
                                   _dtype_code(a.dtype), _dtype_code(out.dtype), PREC[precision],
                                   al, bl, ctypes.c_void_p(s.cuda_stream))
        _check(code, "gemm_run_host")
        return out

    def plan(self, a, b, out=None, out_dtype=None, precision="default", sm_count=None):
        """The planner's decision for these operands (host-only, nothing launched); by
        default for this handle's device's SM count."""
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(self.device).multi_processor_count
        return plan(a, b, out=out, out_dtype=out_dtype, precision=precision,
                    sm_count=sm_count, handle=self)


def plan_strided(a, b, out=None, out_dtype=None, precision="default", sm_count=148,
                 handle=None):
    """Host-only query of gemm_run_strided's decisions for these views (works without a
    GPU): (plan dict, strided-info dict)."""
    M, K = a.shape
    N = b.shape[1]
    od = _dtype_code(out_dtype) if out_dtype is not None else _dtype_code(a.dtype)
    if out is None:
        out = torch.empty((M, N), dtype=_TORCH_OF[od])
    info, sinfo = PlanInfo(), StridedInfo()
    h = handle.handle if handle is not None else None
    code = lib().gemm_plan_strided(h, M, N, K, ctypes.c_void_p(a.data_ptr()), a.stride(0),
                                   a.stride(1), ctypes.c_void_p(b.data_ptr()), b.stride(0),
                                   b.stride(1), ctypes.c_void_p(out.data_ptr()), out.stride(0),
                                   out.stride(1), _dtype_code(a.dtype), _dtype_code(out.dtype),
                                   PREC[precision], sm_count, ctypes.byref(info),
                                   ctypes.byref(sinfo))
    _check(code, "gemm_plan_strided")
    return info.as_dict(), sinfo.as_dict()


# Stand-in address of C for a plan made without an output tensor: 16-byte aligned and
# outside any process's address space, so the planner's check that C does not overlap A or
# B cannot be set off by where A and B happen to live.
_NO_C = 1 << 62


def plan(a, b, out=None, out_dtype=None, precision="default", sm_count=148, handle=None,
         a_ptr=None, b_ptr=None, c_ptr=None, ldc=None):
    """Host-only planner query (works without a GPU); returns a dict.

    Pointers default to the tensors' data pointers; pass integers to ask about
    alignments the tensors do not have.
    """
    M, K = a.shape
    N = b.shape[1]
    al, lda = operand_layout(a)
    bl, ldb = operand_layout(b)
    od = _dtype_code(out_dtype) if out_dtype is not None else (
        _dtype_code(out.dtype) if out is not None else _dtype_code(a.dtype))
    if ldc is None:
        ldc = max(out.stride(0), N, 1) if out is not None else max(N, 1)
    if c_ptr is None:
        c_ptr = out.data_ptr() if out is not None else _NO_C
    info = PlanInfo()
    code = lib().gemm_plan(handle.handle if handle is not None else None, M, N, K,
                           ctypes.c_void_p(a.data_ptr() if a_ptr is None else a_ptr), lda,
                           ctypes.c_void_p(b.data_ptr() if b_ptr is None else b_ptr), ldb,
                           ctypes.c_void_p(c_ptr), ldc, _dtype_code(a.dtype), od,
                           PREC[precision], al, bl, int(sm_count or 148), ctypes.byref(info))
    _check(code, "gemm_plan")
    return info.as_dict()


_handles = {}


def handle(device=None):
    """The per-device default handle (created on first use)."""
    dev = torch.cuda.current_device() if device is None else int(device)
    h = _handles.get(dev)
    if h is None:
        h = _handles[dev] = Gemm(dev)
    return h


def matmul(a, b, out=None, out_dtype=None, precision="default"):
    """C = a @ b with the default handle of a's device; see :meth:`Gemm.matmul`."""
    return handle(a.device.index).matmul(a, b, out=out, out_dtype=out_dtype, precision=precision)


def softmax_rows(x, out=None, out_dtype=None):
    """Row softmax with the default handle of x's device; see :meth:`Gemm.softmax_rows`."""
    return handle(x.device.index).softmax_rows(x, out=out, out_dtype=out_dtype)


def matmul_host(a, b, out=None, out_dtype=None, precision="default", device=None):
    """End-to-end product of host tensors with the default handle of ``device`` (default:
    the current device); see :meth:`Gemm.matmul_host`."""
    dev = torch.cuda.current_device() if device is None else int(device)
    return handle(dev).matmul_host(a, b, out=out, out_dtype=out_dtype, precision=precision)


class Segment(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int32), ("kb_begin", ctypes.c_int32),
                ("kb_end", ctypes.c_int32), ("role", ctypes.c_int32),
                ("first_src", ctypes.c_int32), ("last_src", ctypes.c_int32)]


def schedule(tiles, k_blocks, slots, stream_k=True):
    """Host-only tile schedule: per worker, (whole tiles, [split pieces as tuples])."""
    out = []
    for s in range(slots):
        whole = ctypes.c_int32()
        n = lib().gemm_schedule_segments(tiles, k_blocks, slots, int(stream_k), s,
                                         ctypes.byref(whole), None, 0)
        if n < 0:
            raise ValueError("invalid schedule arguments")
        buf = (Segment * max(n, 1))()
        lib().gemm_schedule_segments(tiles, k_blocks, slots, int(stream_k), s,
                                     ctypes.byref(whole), buf, n)
        out.append((whole.value, [(x.tile, x.kb_begin, x.kb_end, x.role, x.first_src,
                                   x.last_src) for x in buf[:n]]))
    return out


def version():
    return lib().gemm_version().decode()
