"""Python binding of the pipelined GEMM C ABI (``include/pipelined_gemm.h``).

Argument marshalling only: every step of the GEMM runs in the CUDA library
``_build/libpipelined_gemm.so``.  PyTorch supplies device memory and streams.
There is no fallback of any kind: if the library is missing or a call fails,
an exception says so.

    import torch, async_copy_pipelined_gb300 as pg
    C = pg.gemm_f32(A, B, fill="tma", stages=4)          # A, B CUDA float32
    C = pg.gemm_bf16(Ab, Bb)                              # A, B CUDA bfloat16
    C = pg.gemm_f32(A_cpu, B_cpu, fill="cpasync")         # host tensors: copied in and out

Leading dimensions come from the tensors' row strides, so a padded matrix is
a column slice of a wider buffer (``buf[:, :K]`` with ``buf.stride(0) == lda``).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "FILL", "OPTIONS", "GemmError", "lib", "library_path", "gemm_f32", "gemm_bf16", "plan_f32", "plan_bf16",
    "device_status", "selftest_bounded_wait", "testing_set_hooks", "status_string", "build",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpipelined_gemm.so")

FILL = {"sync": 0, "cpasync": 1, "tma": 2, "cpasync_mbar": 3, "cpasync_ws": 4}
# Cache-qualifier options (include/pipelined_gemm.h, GEMM_OPT_*), OR-ed into
# the fill code: pass e.g. fill="cpasync", options=("l2_prefetch_128b",).
OPTIONS = {"l2_prefetch_128b": 0x100, "a_evict_first": 0x200, "a_evict_last": 0x400, "b_evict_first": 0x800,
           "b_evict_last": 0x1000}
# GEMM_OPT_ACCUMULATE: FP32 tiles start from C's values (gemm_f32(accumulate=True)).
OPT_ACCUMULATE = 0x2000

GEMM_OK = 0
GEMM_ERR_TIMEOUT = 6
STATUS_NAMES = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_MISALIGNED", 3: "GEMM_ERR_UNSUPPORTED",
                4: "GEMM_ERR_ARCH", 5: "GEMM_ERR_CUDA", 6: "GEMM_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


class GemmPlan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "fill_mode", "block_m", "block_n", "block_k", "thread_m", "thread_n", "threads", "stages",
        "a_copy_bytes", "b_copy_bytes", "smem_bytes", "grid_x", "grid_y", "k_slices", "options",
        "persistent_ctas", "workspace_bytes", "wide_rows")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force)


def _bind(l):
    I, P, U = ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint)
    l.gemm_f32.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, P]
    l.gemm_f32.restype = I
    l.gemm_f32_ws.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, P, ctypes.c_size_t, P]
    l.gemm_f32_ws.restype = I
    l.gemm_f32_noalloc.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, P]
    l.gemm_f32_noalloc.restype = I
    l.gemm_f32_plan.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, ctypes.POINTER(GemmPlan)]
    l.gemm_f32_plan.restype = I
    l.gemm_bf16.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, P]
    l.gemm_bf16.restype = I
    l.gemm_bf16_plan.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, ctypes.POINTER(GemmPlan)]
    l.gemm_bf16_plan.restype = I
    l.gemm_status_string.argtypes = [I]
    l.gemm_status_string.restype = ctypes.c_char_p
    l.gemm_device_status.argtypes = [P, U]
    l.gemm_device_status.restype = I
    l.gemm_selftest_bounded_wait.argtypes = [I, P]
    l.gemm_selftest_bounded_wait.restype = I
    l.gemm_version.argtypes = []
    l.gemm_version.restype = I
    l.gemm_testing_set_hooks.argtypes = [ctypes.c_ulonglong, I]
    l.gemm_testing_set_hooks.restype = I
    l.gemm_testing_withhold_handover.argtypes = [I]
    l.gemm_testing_withhold_handover.restype = I
    l.gemm_testing_f32_wide.argtypes = [I]
    l.gemm_testing_f32_wide.restype = I
    l.gemm_testing_f32_wide_rows.argtypes = [I, I, I, I, I]
    l.gemm_testing_f32_wide_rows.restype = I
    l.gemm_testing_f32_piece.argtypes = [I, I, I, I, I, I, ctypes.POINTER(ctypes.c_int)]
    l.gemm_testing_f32_piece.restype = I
    l.gemm_f32_host.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, P, ctypes.c_size_t, P, P]
    l.gemm_bf16_ws.argtypes = [I, I, I, P, I, P, I, P, I, I, I, I, P, ctypes.c_size_t, P]
    l.gemm_bf16_ws.restype = I
    l.gemm_f32_host.restype = I
    l.gemm_f32_host_scratch.argtypes = [I, I, I, ctypes.POINTER(ctypes.c_size_t)]
    l.gemm_f32_host_scratch.restype = I
    IP = ctypes.POINTER(ctypes.c_int)
    l.gemm_f32_host_schedule.argtypes = [I, I, I, I, IP, I, IP, IP, I, IP]
    l.gemm_f32_host_schedule.restype = I
    l.gemm_testing_host_policy.argtypes = [I, I, I, I, I, I]
    l.gemm_testing_host_policy.restype = I
    l.gemm_testing_host_streams.argtypes = [I, I, I]
    l.gemm_testing_host_streams.restype = I
    return l


def lib():
    """The loaded C library (ctypes).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"CUDA library not built ({_LIB_PATH} missing): run "
                    "`python -m async_copy_pipelined_gb300.buildlib` or __graft_entry__.build()")
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().gemm_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(status), f"status {status}")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _fill_code(fill, options=()) -> int:
    if isinstance(fill, str):
        if fill not in FILL:
            raise ValueError(f"fill must be one of {sorted(FILL)}")
        code = FILL[fill]
    else:
        code = int(fill)
    for o in options:
        if o not in OPTIONS:
            raise ValueError(f"options must be among {sorted(OPTIONS)}")
        code |= OPTIONS[o]
    return code


def _matrix_args(x, name):
    """(rows, cols, ld, pointer) of a 2-D tensor whose rows are contiguous."""
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if x.numel() == 0:  # an empty matrix has no layout to check (its strides are arbitrary)
        return x.shape[0], x.shape[1], max(x.shape[1], 1), x.data_ptr()
    if x.shape[1] > 1 and x.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride (row-major rows)")
    rows, cols = x.shape
    ld = x.stride(0) if x.stride(0) >= cols else cols
    return rows, cols, max(ld, 1), x.data_ptr()


def _operand_device(A, B, C, stream):
    """The one device A, B and C (if given) all live on; the kernels read and
    write them through raw pointers, so mixed host/device operands or
    operands on two GPUs are refused rather than launched."""
    for name, t in (("B", B), ("C", C)):
        if t is not None and t.device != A.device:
            raise ValueError(f"A is on {A.device} but {name} is on {t.device}: "
                             "all operands must be on one device (or all on the host)")
    dev = A.device
    if dev.type == "cuda" and stream is not None and getattr(stream, "device", dev) != dev:
        raise ValueError(f"stream belongs to {stream.device}, operands to {dev}")
    return dev


def _byte_range(x):
    """[first, last) bytes a row-major 2-D tensor view spans."""
    rows, cols = x.shape
    if rows == 0 or cols == 0:
        return (0, 0)
    first = x.data_ptr()
    return first, first + ((rows - 1) * x.stride(0) + cols) * x.element_size()


def _refuse_aliased_output(C, A, B):
    """C is written while other blocks still read A and B: an output that
    shares bytes with an input would give wrong results, so it is refused."""
    c0, c1 = _byte_range(C)
    for name, t in (("A", A), ("B", B)):
        t0, t1 = _byte_range(t)
        if c0 < t1 and t0 < c1:
            raise ValueError(f"C overlaps {name} in memory; the output must not alias an input")


def _check(status: int, what: str):
    if status != GEMM_OK:
        raise GemmError(status, what)


def plan_f32(M, N, K, lda=None, ldb=None, ldc=None, fill="tma", stages=0, block_tile=0,
             a_ptr=256, b_ptr=256, c_ptr=256, options=()) -> dict:
    """What gemm_f32 would launch for these sizes (no device access)."""
    p = GemmPlan()
    st = lib().gemm_f32_plan(M, N, K, a_ptr, lda or max(K, 1), b_ptr, ldb or max(N, 1), c_ptr, ldc or max(N, 1),
                             _fill_code(fill, options), stages, block_tile, ctypes.byref(p))
    _check(st, "gemm_f32_plan")
    return p.as_dict()


def plan_bf16(M, N, K, lda=None, ldb=None, ldc=None, fill="tma", stages=0, block_m=0, a_ptr=256, b_ptr=256,
              c_ptr=256, options=()) -> dict:
    p = GemmPlan()
    st = lib().gemm_bf16_plan(M, N, K, a_ptr, lda or max(K, 1), b_ptr, ldb or max(N, 1), c_ptr, ldc or max(N, 1),
                              _fill_code(fill, options), stages, block_m, ctypes.byref(p))
    _check(st, "gemm_bf16_plan")
    return p.as_dict()


# BF16 host-buffer calls (host tensors in, host C out) run on three streams
# made once per device: one carries the host-to-device copies, one the GEMMs,
# one the device-to-host copies, ordered by events, with C cut into row
# chunks of about HOST_CHUNK_WAVES waves of 128 x 128 tiles so that each
# chunk's copies overlap the GEMMs of others.  FP32 host-buffer calls go to
# the library's native executor instead (gemm_f32_host in the C header).
HOST_CHUNK_WAVES = 1.25
HOST_CHUNK_MIN_ROWS = 256
HOST_STREAMS = 3
_host_streams = {}
_host_sms = {}
_host_scratch = {}
_host_status = {}


def host_chunk_rows(N: int, sms: int) -> int:
    """Rows per chunk of the BF16 host path: enough 128 x 128 tiles for
    HOST_CHUNK_WAVES waves on `sms` SMs, a multiple of 256 rows (whole tiles
    of every kernel), at least HOST_CHUNK_MIN_ROWS."""
    tiles_n = max(1, -(-N // 128))
    tile_rows = -(-int(HOST_CHUNK_WAVES * sms) // tiles_n)
    rows = max(HOST_CHUNK_MIN_ROWS, tile_rows * 128)
    return -(-rows // 256) * 256


def host_row_chunks(M: int, N: int, sms: int = 152):
    """Row ranges [r0, r1) of the BF16 host path, in order."""
    rows = host_chunk_rows(N, sms)
    return [(r0, min(M, r0 + rows)) for r0 in range(0, M, rows)]


def host_schedule_f32(M: int, N: int, K: int, sms: int = 152):
    """The cut the native FP32 host-buffer executor makes (no device is
    touched): (K-block bounds, row-chunk bounds of the last block)."""
    kb = (ctypes.c_int * 17)()
    rb = (ctypes.c_int * 65)()
    nk, nr = ctypes.c_int(), ctypes.c_int()
    st = lib().gemm_f32_host_schedule(M, N, K, sms, kb, 17, ctypes.byref(nk), rb, 65, ctypes.byref(nr))
    _check(st, "gemm_f32_host_schedule")
    return list(kb[: nk.value + 1]), list(rb[: nr.value + 1])


def _streams_for(dev):
    import torch
    streams = _host_streams.get(dev.index)
    if streams is None:
        streams = _host_streams[dev.index] = [torch.cuda.Stream(dev) for _ in range(HOST_STREAMS)]
    return streams


def _sms_of(dev) -> int:
    import torch
    n = _host_sms.get(dev.index)
    if n is None:
        n = _host_sms[dev.index] = torch.cuda.get_device_properties(dev).multi_processor_count
    return n


def _f32_host_call(A, B, C, code, stages, block_tile):
    """FP32 host tensors through the native executor (gemm_f32_host): the
    device copies and the K-split hand-over space live in a scratch buffer
    kept per device and grown as needed (the executor serialises its calls
    on a device, so one buffer serves them all).  Returns once C is on the
    host and the device status word has been checked."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    M, K, lda, pa = _matrix_args(A, "A")
    K2, N, ldb, pb = _matrix_args(B, "B")
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {M}x{K}, B is {K2}x{N}")
    if A.dtype != torch.float32 or B.dtype != torch.float32:
        raise TypeError("gemm_f32 takes float32 tensors")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    Mc, Nc, ldc, pc = _matrix_args(C, "C")
    if (Mc, Nc) != (M, N) or C.dtype != torch.float32:
        raise ValueError("C must be a float32 M x N tensor")
    need = ctypes.c_size_t()
    _check(lib().gemm_f32_host_scratch(M, N, K, ctypes.byref(need)), "gemm_f32_host_scratch")
    scratch = _host_scratch.get(dev.index)
    if scratch is None or scratch.numel() < need.value:
        _host_scratch.pop(dev.index, None)
        scratch = _host_scratch[dev.index] = torch.empty(max(need.value, 256), dtype=torch.uint8, device=dev)
    word = _host_status.get(dev.index)
    if word is None:
        word = _host_status[dev.index] = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    cur = torch.cuda.current_stream(dev)
    st = lib().gemm_f32_host(M, N, K, pa, lda, pb, ldb, pc, ldc, code, stages, block_tile, scratch.data_ptr(),
                             scratch.numel(), word.data_ptr(), ctypes.c_void_p(cur.cuda_stream))
    cur.synchronize()  # whatever was enqueued, even after an error, is done
    _check(st, "gemm_f32_host")
    # The executor copied the status word out after its last GEMM: a kernel
    # that gave up on a bounded wait left its rows of C undefined.
    detail = ctypes.c_uint32.from_address(word.data_ptr()).value
    if detail:
        _check(GEMM_ERR_TIMEOUT, f"host-buffer GEMM (device status word {detail:#x})")
    return C


def _host_roundtrip(fn, A, B, C, dtype_out):
    """BF16 host tensors in, host C out.

    fn(a, b, c, stream) runs the library's GEMM on device tensors, writing c.
    Copies in, GEMMs and copies out each run in order on a stream of their
    own: B first, then each row chunk's rows of A, its GEMM as soon as they
    have landed, and its rows of C copied out as soon as the GEMM is done.
    Each C element is computed from the same row of A, the same B and the
    same arithmetic as in a single call, so the cutting changes no result
    bit.  Host tensors should be pinned for the copies to be asynchronous.
    The device buffers are allocated on the caller's current stream and held
    until the call has synchronised, so no other work reuses them while the
    side streams do.  Returns after C has been written."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    M, K, N = A.shape[0], A.shape[1], B.shape[1]
    if C is None:
        C = torch.empty((M, N), dtype=dtype_out, pin_memory=True)
    cur = torch.cuda.current_stream(dev)
    h2d, comp, d2h = _streams_for(dev)
    Ad = torch.empty((M, K), dtype=A.dtype, device=dev)
    Bd = torch.empty((K, N), dtype=B.dtype, device=dev)
    Cd = torch.empty((M, N), dtype=dtype_out, device=dev)

    def mark(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    start = mark(cur)  # the side streams begin after what `cur` already holds
    for s in (h2d, comp, d2h):
        s.wait_event(start)
    with torch.cuda.stream(h2d):
        Bd.copy_(B, non_blocking=True)
    for r0, r1 in host_row_chunks(M, N, _sms_of(dev)):
        with torch.cuda.stream(h2d):
            Ad[r0:r1].copy_(A[r0:r1], non_blocking=True)
        comp.wait_event(mark(h2d))  # this chunk's rows of A, and all of B before them
        with torch.cuda.stream(comp):
            fn(Ad[r0:r1], Bd, Cd[r0:r1], comp)
        d2h.wait_event(mark(comp))
        with torch.cuda.stream(d2h):
            C[r0:r1].copy_(Cd[r0:r1], non_blocking=True)
    for s in (h2d, comp, d2h):
        cur.wait_stream(s)
    cur.synchronize()
    # Every GEMM is ordered before this point of `cur`: a kernel that gave up
    # on a bounded wait left its rows of C undefined.
    st, detail = device_status(cur)
    _check(st, f"host-buffer GEMM (device status word {detail:#x})")
    return C


# Hand-over workspaces of gemm_f32_ws, one per (device, stream): a workspace
# serves one call at a time, and calls on one stream never overlap.
_workspaces = {}


def _workspace(dev, stream_handle: int, nbytes: int):
    import torch
    key = (dev.index, stream_handle)
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = _workspaces[key] = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    return buf


def gemm_f32(A, B, C=None, *, fill="tma", stages=0, block_tile=0, stream=None, options=(), workspace="auto",
             accumulate=False):
    """C = A @ B in float32 through the library's FP32 kernel with the given fill.

    A (M x K), B (K x N) float32 tensors; C (M x N) float32 output, allocated
    if None.  CUDA tensors run on the device asynchronously on `stream`
    (default: torch's current stream).  CPU tensors go through the native
    host-buffer executor (gemm_f32_host in the C header): B's rows and A's
    columns cross the link in K blocks, each block's GEMM starts as soon as
    it has landed and continues the FMA chains of the block before it, and
    the last block's row chunks are copied out as they finish; the workspace
    argument does not apply (the executor keeps its own).  The call returns
    once C is on the host, after the device status word has been checked
    (GemmError on a kernel timeout).

    options: cache-qualifier names from OPTIONS (GEMM_OPT_* in the C
    header): an L2 prefetch size for cp.async copies and L2 eviction
    priorities for A and B; none changes a result bit.

    accumulate: C = C + A @ B, each element's FMA chain continuing from the
    value C holds (GEMM_OPT_ACCUMULATE): a call over the first K0 columns
    of A and rows of B followed by an accumulating call over the rest gives
    the bits of one call over all K.  Needs C; device tensors only.

    workspace: hand-over space for the persistent TMA kernel's split of the
    last round of tiles (gemm_f32_ws in the C header).  "auto" keeps one
    buffer per device and stream, grown as needed; None runs without the
    split; a uint8 CUDA tensor is used as given.  The bits are the same
    either way.

    The device path returns as soon as the kernel is enqueued.  Its C is known
    good only once device_status() has returned status 0 for a point after
    the call: a kernel that gave up on a bounded wait leaves C undefined and
    records GEMM_ERR_TIMEOUT in the device's status word instead.
    """
    import torch
    dev = _operand_device(A, B, C, stream)
    if not A.is_cuda:
        if C is not None:
            _refuse_aliased_output(C, A, B)
        if accumulate:
            raise ValueError("accumulate takes device tensors")
        # block_tile 0: the executor picks the whole problem's tile.
        return _f32_host_call(A, B, C, _fill_code(fill, options), stages, block_tile)
    if A.dtype != torch.float32 or B.dtype != torch.float32:
        raise TypeError("gemm_f32 takes float32 tensors")
    M, K, lda, pa = _matrix_args(A, "A")
    K2, N, ldb, pb = _matrix_args(B, "B")
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {M}x{K}, B is {K2}x{N}")
    if C is None:
        if accumulate:
            raise ValueError("accumulate needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
    Mc, Nc, ldc, pc = _matrix_args(C, "C")
    if (Mc, Nc) != (M, N) or C.dtype != torch.float32:
        raise ValueError("C must be a float32 M x N tensor")
    _refuse_aliased_output(C, A, B)
    code = _fill_code(fill, options) | (OPT_ACCUMULATE if accumulate else 0)
    with torch.cuda.device(dev):
        sh = _stream_handle(stream)
        ws_ptr, ws_bytes = None, 0
        if workspace is not None:
            plan = GemmPlan()
            st = lib().gemm_f32_plan(M, N, K, pa, lda, pb, ldb, pc, ldc, code, stages, block_tile, ctypes.byref(plan))
            _check(st, "gemm_f32_plan")
            if plan.workspace_bytes > 0:
                ws = _workspace(dev, sh.value or 0, plan.workspace_bytes) if isinstance(workspace, str) else workspace
                if ws.device != dev:
                    raise ValueError(f"workspace is on {ws.device}, operands on {dev}")
                ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
        st = lib().gemm_f32_ws(M, N, K, pa, lda, pb, ldb, pc, ldc, code, stages, block_tile, ws_ptr, ws_bytes, sh)
    _check(st, "gemm_f32")
    return C


def gemm_bf16(A, B, C=None, *, fill="tma", stages=0, block_m=0, stream=None, options=(), workspace=None):
    """C (float32) = A @ B for bfloat16 A (M x K), B (K x N) on the tensor cores.

    fill: "tma" (default), "cpasync" or "sync" fills the shared-memory stages
    the MMAs read; block_m: 128 or 256 rows per CTA tile, 0 to let the
    library choose.  Every fill and tile gives the same bits.  workspace:
    hand-over space for the TMA fill's K split of the last round of tiles
    (gemm_bf16_ws in the C header), as for gemm_f32: None (the default: no
    split), "auto" or a uint8 CUDA tensor; the bits are the same either
    way.  The split is off by default because on GB300 it measured slower
    than the unsplit kernel at 8192^3 (603 against 584 us on the 256-row
    tile): its extra accumulator drains cost more than the idle SMs of the
    partial last round.  Host
    tensors and the device status word are handled as in gemm_f32: on the
    device path, check device_status() before trusting C."""
    import torch
    dev = _operand_device(A, B, C, stream)
    if not A.is_cuda:
        if C is not None:
            _refuse_aliased_output(C, A, B)
        if block_m == 0:
            # The tile the whole problem would get, not what one row chunk
            # alone would get.
            M, K, N = A.shape[0], A.shape[1], B.shape[1]
            try:
                block_m = plan_bf16(M, N, K, lda=(K + 7) // 8 * 8, ldb=(N + 7) // 8 * 8, fill=fill,
                                    stages=stages)["block_m"]
            except (RuntimeError, ValueError):
                pass  # the chunk calls report the error
        return _host_roundtrip(lambda a, b, c, s: gemm_bf16(a, b, c, fill=fill, stages=stages, block_m=block_m,
                                                            stream=s, options=options, workspace=workspace),
                               A, B, C, torch.float32)
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("gemm_bf16 takes bfloat16 tensors")
    M, K, lda, pa = _matrix_args(A, "A")
    K2, N, ldb, pb = _matrix_args(B, "B")
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {M}x{K}, B is {K2}x{N}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
    Mc, Nc, ldc, pc = _matrix_args(C, "C")
    if (Mc, Nc) != (M, N) or C.dtype != torch.float32:
        raise ValueError("C must be a float32 M x N tensor")
    _refuse_aliased_output(C, A, B)
    code = _fill_code(fill, options)
    with torch.cuda.device(dev):
        sh = _stream_handle(stream)
        ws_ptr, ws_bytes = None, 0
        if workspace is not None:
            plan = GemmPlan()
            st = lib().gemm_bf16_plan(M, N, K, pa, lda, pb, ldb, pc, ldc, code, stages, block_m, ctypes.byref(plan))
            _check(st, "gemm_bf16_plan")
            if plan.workspace_bytes > 0:
                ws = _workspace(dev, sh.value or 0, plan.workspace_bytes) if isinstance(workspace, str) else workspace
                if ws.device != dev:
                    raise ValueError(f"workspace is on {ws.device}, operands on {dev}")
                ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
        st = lib().gemm_bf16_ws(M, N, K, pa, lda, pb, ldb, pc, ldc, code, stages, block_m, ws_ptr, ws_bytes, sh)
    _check(st, "gemm_bf16")
    return C


def device_status(stream=None):
    """(status, detail word) after synchronising `stream`; clears the word.

    The word is one per device, shared by all streams: it covers the work
    ordered before this point of `stream`, and a kernel on another stream can
    record (or have its record cleared) concurrently."""
    detail = ctypes.c_uint(0)
    st = lib().gemm_device_status(_stream_handle(stream), ctypes.byref(detail))
    return st, detail.value


def selftest_bounded_wait(timeout_us: int, stream=None) -> int:
    return lib().gemm_selftest_bounded_wait(int(timeout_us), _stream_handle(stream))


def testing_set_hooks(wait_limit_ns: int = 0, withhold: int = -1) -> None:
    """Test hooks (include/pipelined_gemm_testing.h): the GEMM kernels' wait
    limit (0: the default 2 s) and a ring position their producers leave
    unfilled (-1: none), for every later call in this process."""
    _check(lib().gemm_testing_set_hooks(int(wait_limit_ns), int(withhold)), "gemm_testing_set_hooks")


def testing_f32_wide(mode: int = -1) -> None:
    """How later FP32 TMA calls on the 128 tile pick their wide rows
    (include/pipelined_gemm_testing.h): -1 by the cost model, 0 never,
    1 whenever a cut exists.  The bits are the same in every mode."""
    _check(lib().gemm_testing_f32_wide(int(mode)), "gemm_testing_f32_wide")


def f32_wide_rows(M: int, N: int, K: int, sms: int = 152, mode: int = -1) -> int:
    """Rows [0, r) of an M x N x K TMA call on the 128 tile that the
    128 x 256 wide-row kernel computes (computed on the host)."""
    r = lib().gemm_testing_f32_wide_rows(int(M), int(N), int(K), int(sms), int(mode))
    if r < 0:
        raise ValueError("invalid arguments")
    return r
