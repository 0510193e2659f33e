"""Python binding of libpurlin1 (include/purlin.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
computation of its own: all data movement happens in the library's CUDA
kernels.  If the shared library has not been built, importing this module
raises ImportError -- there is no fallback path.

Conventions: buffers are passed as device pointers (``tensor.data_ptr()``);
streams as raw ``cudaStream_t`` values (``torch.cuda.current_stream().cuda_stream``).
Creators return opaque handles; calls that fail raise ``PurlinError`` carrying
the ``pl_status`` code, except ``pl_ctx_status`` which returns the code (a
timeout is an expected answer there).
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpurlin1.so")

PL_OK, PL_ERR_INVALID, PL_ERR_LAYOUT, PL_ERR_ALIAS = 0, 1, 2, 3
PL_ERR_NOMEM, PL_ERR_CUDA, PL_ERR_TIMEOUT, PL_ERR_UNSUPPORTED = 4, 5, 6, 7
PL_COPY, PL_SUM, PL_MAX = 0, 1, 2
PL_BF16, PL_FP32, PL_FP16, PL_FP8 = 0, 1, 2, 3
PL_PATH_AUTO, PL_PATH_ZS, PL_PATH_STAGED = 0, 1, 2
PL_AR_AUTO, PL_AR_FUSED, PL_AR_COMPOSED, PL_AR_NOTIFIED = 0, 1, 2, 3
PL_ATOM_AUTO, PL_ATOM_VECTOR, PL_ATOM_BULK, PL_ATOM_INLINE = 0, 1, 2, 3
PL_ITEM_MOVE, PL_ITEM_STAGE, PL_ITEM_CONSUME, PL_ITEM_COMPOSE = 0, 1, 2, 3
PL_SPACE_IN, PL_SPACE_OUT, PL_SPACE_SCRATCH = 0, 1, 2
PL_SYNC_WAIT_FULL, PL_SYNC_WAIT_FREE, PL_SYNC_NOTIFY, PL_SYNC_CREDIT = 0, 1, 2, 3

DTYPES = {"bf16": PL_BF16, "fp32": PL_FP32, "fp16": PL_FP16, "fp8": PL_FP8}
OPS = {"copy": PL_COPY, "sum": PL_SUM, "max": PL_MAX}


class PurlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pl_status_str(status)} (pl_status {status})")


class pl_part(C.Structure):
    _fields_ = [("name", C.c_uint64), ("offset", C.c_uint64), ("len", C.c_uint64),
                ("rows", C.c_uint64), ("row_stride", C.c_uint64)]


class pl_policy(C.Structure):
    _fields_ = [("path", C.c_int32), ("allreduce_form", C.c_int32), ("datapath", C.c_int32),
                ("ctas", C.c_int32), ("stages", C.c_int32), ("reserved0", C.c_int32),
                ("chunk_bytes", C.c_uint64), ("poll_timeout_ns", C.c_uint64),
                ("debug_drop_notify", C.c_int64)]


class pl_plan_stats(C.Structure):
    _fields_ = [("items", C.c_uint64), ("refs", C.c_uint64), ("syncs", C.c_uint64),
                ("flags", C.c_uint64), ("chunk_elems", C.c_uint64), ("slots", C.c_uint64),
                ("slot_elems", C.c_uint64), ("ctas", C.c_int32), ("threads", C.c_int32),
                ("uses_tickets", C.c_int32), ("path", C.c_int32),
                ("bytes_read", C.c_uint64), ("bytes_written", C.c_uint64),
                ("datapath", C.c_int32), ("reserved0", C.c_int32)]


class pl_plan_item(C.Structure):
    _fields_ = [("kind", C.c_int32), ("op", C.c_int32), ("nsrc", C.c_int32), ("ndst", C.c_int32),
                ("nwait", C.c_int32), ("npost", C.c_int32), ("rows", C.c_uint64), ("cols", C.c_uint64)]


class pl_plan_ref(C.Structure):
    _fields_ = [("space", C.c_int32), ("index", C.c_int32), ("offset", C.c_uint64), ("stride", C.c_uint64)]


class pl_plan_sync(C.Structure):
    _fields_ = [("type", C.c_int32), ("flag", C.c_uint32), ("use", C.c_uint32), ("count", C.c_uint32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpurlin1 is not built ({LIB_PATH} is missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = C.CDLL(LIB_PATH)
    vp, u64, i32 = C.c_void_p, C.c_uint64, C.c_int32
    u64p, vpp, intp = C.POINTER(C.c_uint64), C.POINTER(C.c_void_p), C.POINTER(C.c_int)
    sig = {
        "pl_abi_version": (C.c_int, []),
        "pl_status_str": (C.c_char_p, [i32]),
        "pl_policy_default": (None, [C.POINTER(pl_policy)]),
        "pl_layout_create": (i32, [vpp, C.c_int, intp, C.POINTER(pl_part)]),
        "pl_layout_destroy": (i32, [vp]),
        "pl_layout_info": (i32, [vp, intp, intp]),
        "pl_layout_rank_owned": (i32, [vpp, C.c_int, u64p]),
        "pl_layout_partitioned": (i32, [vpp, C.c_int, u64p]),
        "pl_layout_rank_owned_inplace": (i32, [vpp, C.c_int, u64p]),
        "pl_layout_alltoall_in": (i32, [vpp, C.c_int, u64p]),
        "pl_layout_alltoall_out": (i32, [vpp, C.c_int, u64p]),
        "pl_layout_ulysses_in": (i32, [vpp, C.c_int, u64, u64, u64]),
        "pl_layout_ulysses_out": (i32, [vpp, C.c_int, u64, u64, u64]),
        "pl_ctx_create": (i32, [vpp, C.c_int, u64]),
        "pl_ctx_destroy": (i32, [vp]),
        "pl_ctx_status": (i32, [vp, vp]),
        "pl_ctx_cuda_error": (C.c_int, [vp]),
        "pl_ctx_launches": (u64, [vp]),
        "pl_collective": (i32, [vp, vp, vp, i32, i32, C.c_int, vpp, u64p, vpp, u64p,
                                C.POINTER(pl_policy), vp]),
        "pl_allreduce": (i32, [vp, i32, C.c_int, u64, vpp, vpp, C.POINTER(pl_policy), vp]),
        "pl_allreduce_op": (i32, [vp, i32, i32, C.c_int, u64, vpp, vpp, C.POINTER(pl_policy), vp]),
        "pl_allreduce_noalloc": (i32, [i32, C.c_int, u64, vpp, vpp, C.c_int, vp]),
        "pl_plan_create": (i32, [vpp, vp, vp, i32, i32, C.c_int, C.POINTER(pl_policy), C.c_int, u64]),
        "pl_plan_destroy": (i32, [vp]),
        "pl_plan_get_stats": (i32, [vp, C.POINTER(pl_plan_stats)]),
        "pl_plan_get_item": (i32, [vp, u64, C.POINTER(pl_plan_item), C.POINTER(pl_plan_ref), C.c_int,
                                   C.POINTER(pl_plan_sync), C.c_int]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def _check(st: int, where: str) -> None:
    if st != PL_OK:
        raise PurlinError(st, where)


def _u64s(xs):
    xs = [int(x) for x in xs]
    return (C.c_uint64 * max(1, len(xs)))(*xs)


def _ptrs(ps):
    arr = (C.c_void_p * max(1, len(ps)))()
    for i, p in enumerate(ps):
        arr[i] = int(p) if p else None
    return arr


def _dtype(dt) -> int:
    return DTYPES[dt] if isinstance(dt, str) else int(dt)


def _op(op) -> int:
    return OPS[op] if isinstance(op, str) else int(op)


# ------------------------------------------------------------------- misc


def pl_abi_version() -> int:
    return lib.pl_abi_version()


def pl_status_str(st: int) -> str:
    return lib.pl_status_str(int(st)).decode()


def pl_policy_default(**overrides) -> pl_policy:
    """The all-auto policy, with the named fields overridden."""
    p = pl_policy()
    lib.pl_policy_default(C.byref(p))
    for k, v in overrides.items():
        setattr(p, k, v)
    return p


# ------------------------------------------------------------ owned handles


class Handle(int):
    """An opaque library handle: an int, as the C calls take it, that owns the
    object behind it.  The object is freed by its destroy call or, failing
    that, when the handle is garbage-collected; freeing twice is a no-op."""

    _destroy_name = ""

    def __new__(cls, value: int):
        h = super().__new__(cls, value)
        h._live = True
        return h

    def release(self) -> None:
        if self._live:
            self._live = False
            _check(getattr(lib, self._destroy_name)(int(self)), self._destroy_name)

    def __del__(self):
        if getattr(self, "_live", False):
            self._live = False
            try:
                getattr(lib, self._destroy_name)(int(self))
            except Exception:  # interpreter shutdown: the library may be gone
                pass


class Layout(Handle):
    _destroy_name = "pl_layout_destroy"


class Plan(Handle):
    _destroy_name = "pl_plan_destroy"


# ---------------------------------------------------------------- layouts


def pl_layout_create(R: int, parts_per_rank) -> int:
    """parts_per_rank[r]: list of (name, offset, len) or (name, offset, len, rows, row_stride)."""
    counts = (C.c_int * R)(*[len(p) for p in parts_per_rank])
    flat = []
    for parts in parts_per_rank:
        for p in parts:
            p = tuple(int(v) for v in p)
            if len(p) == 3:
                p = p + (1, p[2])
            flat.append(pl_part(*p))
    arr = (pl_part * max(1, len(flat)))(*flat)
    h = C.c_void_p()
    _check(lib.pl_layout_create(C.byref(h), R, counts, arr), "pl_layout_create")
    return Layout(h.value)


def pl_layout_destroy(layout: int) -> None:
    if isinstance(layout, Handle):
        layout.release()
    else:
        _check(lib.pl_layout_destroy(layout), "pl_layout_destroy")


def pl_layout_info(layout: int):
    R, n = C.c_int(), C.c_int()
    _check(lib.pl_layout_info(layout, C.byref(R), C.byref(n)), "pl_layout_info")
    return R.value, n.value


def _builder(name):
    def make(R: int, lens) -> int:
        h = C.c_void_p()
        _check(getattr(lib, name)(C.byref(h), R, _u64s(lens)), name)
        return Layout(h.value)
    make.__name__ = name
    make.__doc__ = f"Calls {name}(R, lens) and returns the layout handle."
    return make


pl_layout_rank_owned = _builder("pl_layout_rank_owned")
pl_layout_partitioned = _builder("pl_layout_partitioned")
pl_layout_rank_owned_inplace = _builder("pl_layout_rank_owned_inplace")


def pl_layout_alltoall_in(R: int, lens_matrix) -> int:
    h = C.c_void_p()
    _check(lib.pl_layout_alltoall_in(C.byref(h), R, _u64s([x for row in lens_matrix for x in row])),
           "pl_layout_alltoall_in")
    return Layout(h.value)


def pl_layout_alltoall_out(R: int, lens_matrix) -> int:
    h = C.c_void_p()
    _check(lib.pl_layout_alltoall_out(C.byref(h), R, _u64s([x for row in lens_matrix for x in row])),
           "pl_layout_alltoall_out")
    return Layout(h.value)


def pl_layout_ulysses_in(R: int, S: int, H: int, D: int) -> int:
    h = C.c_void_p()
    _check(lib.pl_layout_ulysses_in(C.byref(h), R, S, H, D), "pl_layout_ulysses_in")
    return Layout(h.value)


def pl_layout_ulysses_out(R: int, S: int, H: int, D: int) -> int:
    h = C.c_void_p()
    _check(lib.pl_layout_ulysses_out(C.byref(h), R, S, H, D), "pl_layout_ulysses_out")
    return Layout(h.value)


# ---------------------------------------------------------------- context


def pl_ctx_create(device: int = 0, scratch_bytes: int = 0) -> int:
    h = C.c_void_p()
    _check(lib.pl_ctx_create(C.byref(h), device, scratch_bytes), "pl_ctx_create")
    return h.value


def pl_ctx_destroy(ctx: int) -> None:
    _check(lib.pl_ctx_destroy(ctx), "pl_ctx_destroy")


def pl_ctx_status(ctx: int, stream: int = 0) -> int:
    """Waits for `stream`; returns PL_OK or the device status (e.g. PL_ERR_TIMEOUT)."""
    return lib.pl_ctx_status(ctx, stream or None)


def pl_ctx_cuda_error(ctx: int) -> int:
    return lib.pl_ctx_cuda_error(ctx)


def pl_ctx_launches(ctx: int) -> int:
    return lib.pl_ctx_launches(ctx)


# ------------------------------------------------------------ collectives


def pl_collective(ctx, in_layout, out_layout, op, dtype, R, in_ptrs, in_counts, out_ptrs, out_counts,
                  policy: pl_policy | None = None, stream: int = 0) -> None:
    st = lib.pl_collective(ctx, in_layout, out_layout, _op(op), _dtype(dtype), R,
                           _ptrs(in_ptrs), _u64s(in_counts), _ptrs(out_ptrs), _u64s(out_counts),
                           C.byref(policy) if policy is not None else None, stream or None)
    _check(st, "pl_collective")


def pl_allreduce(ctx, dtype, R, count, in_ptrs, out_ptrs, policy: pl_policy | None = None,
                 stream: int = 0) -> None:
    st = lib.pl_allreduce(ctx, _dtype(dtype), R, count, _ptrs(in_ptrs), _ptrs(out_ptrs),
                          C.byref(policy) if policy is not None else None, stream or None)
    _check(st, "pl_allreduce")


def pl_allreduce_op(ctx, op, dtype, R, count, in_ptrs, out_ptrs, policy: pl_policy | None = None,
                    stream: int = 0) -> None:
    st = lib.pl_allreduce_op(ctx, _op(op), _dtype(dtype), R, count, _ptrs(in_ptrs), _ptrs(out_ptrs),
                             C.byref(policy) if policy is not None else None, stream or None)
    _check(st, "pl_allreduce_op")


def pl_allreduce_noalloc(dtype, R, count, in_ptrs, out_ptrs, wait: bool = True, stream: int = 0) -> int:
    """AllReduce that allocates no device memory (its state lives in the
    library's static device array).  Returns the pl_status: with wait=True it
    also waits for `stream` and reports a device-side timeout."""
    return lib.pl_allreduce_noalloc(_dtype(dtype), R, count, _ptrs(in_ptrs), _ptrs(out_ptrs), 1 if wait else 0,
                                    stream or None)


# ------------------------------------------------------- plan introspection


def pl_plan_create(in_layout, out_layout, op, dtype, R, policy: pl_policy | None = None,
                   num_sms: int = 152, scratch_bytes: int = 0) -> int:
    h = C.c_void_p()
    _check(lib.pl_plan_create(C.byref(h), in_layout, out_layout, _op(op), _dtype(dtype), R,
                              C.byref(policy) if policy is not None else None, num_sms, scratch_bytes),
           "pl_plan_create")
    return Plan(h.value)


def pl_plan_destroy(plan: int) -> None:
    if isinstance(plan, Handle):
        plan.release()
    else:
        _check(lib.pl_plan_destroy(plan), "pl_plan_destroy")


def pl_plan_get_stats(plan: int) -> pl_plan_stats:
    s = pl_plan_stats()
    _check(lib.pl_plan_get_stats(plan, C.byref(s)), "pl_plan_get_stats")
    return s


def pl_plan_get_item(plan: int, i: int):
    """(pl_plan_item, [pl_plan_ref...], [pl_plan_sync...]) of work item i."""
    it = pl_plan_item()
    _check(lib.pl_plan_get_item(plan, i, C.byref(it), None, 0, None, 0), "pl_plan_get_item")
    nref, nsync = it.nsrc + it.ndst, it.nwait + it.npost
    refs = (pl_plan_ref * max(1, nref))()
    syncs = (pl_plan_sync * max(1, nsync))()
    _check(lib.pl_plan_get_item(plan, i, C.byref(it), refs, nref, syncs, nsync), "pl_plan_get_item")
    return it, list(refs[:nref]), list(syncs[:nsync])


# ------------------------------------------------------------ torch glue


def ptrs(tensors):
    """Device pointers of a list of tensors (None stays None)."""
    return [t.data_ptr() if t is not None else 0 for t in tensors]


def counts(tensors):
    """Element counts of a list of tensors."""
    return [t.numel() if t is not None else 0 for t in tensors]


def stream_handle(stream=None) -> int:
    """Raw cudaStream_t of a torch stream (the current stream by default)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)
