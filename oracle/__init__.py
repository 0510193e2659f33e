"""CPU oracle for the Purlin collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product (``copy_reduce_datapath_gb300``
and its ``libpurlin1``) shares no code with it and never imports it.

The arithmetic lives in ``oracle.c`` (plain C loops, one element at a time);
this module only marshals numpy arrays into it.  Element storage:

* ``"bf16"`` and ``"fp16"`` arrays are ``numpy.uint16`` bit patterns;
* ``"fp32"`` arrays are ``numpy.float32``;
* ``"fp8"`` arrays are ``numpy.uint8`` bytes (any 1-byte format: moved, never reduced).

Every function cites the passage of "Purlin: Separating Orchestration from the
Datapath of Collectives" that it writes out:

========================  ==============================================
``allgather``             Figure 4 caption (AllGather), Table 2 (V form)
``reducescatter``         Figure 4 caption (ReduceScatter), Table 2
``allreduce``             Table 2 (TP AllReduce), Figure 6 caption
``alltoall``              Figure 4 caption (AllToAll), Table 2
``ulysses_a2a``           Table 2, Ulysses row (sequence <-> head)
``collective``            abstract: input layout + output layout + op
``f32_to_bf16``           the output rounding (IEEE round-to-nearest-even)
``f32_to_f16``            the same rounding to IEEE binary16
========================  ==============================================

Parity pins live in ``tests/test_oracle_pins.py``; every function above is
pinned there by something other than itself (hand-written Figure 4
placements, exact integer sums, library routines, invariants, brute force),
and ``tests/test_oracle_mutations.py`` shows that planted mistakes in
``oracle.c`` fail those pins.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build

BF16, FP32, FP16, FP8 = 0, 1, 2, 3
COPY, SUM, MAX = 0, 1, 2
_DT = {"bf16": (BF16, np.uint16), "fp32": (FP32, np.float32), "fp16": (FP16, np.uint16), "fp8": (FP8, np.uint8)}
_OPS = {"copy": COPY, "sum": SUM, "max": MAX}


class _Part(C.Structure):
    _fields_ = [("name", C.c_uint64), ("offset", C.c_uint64), ("len", C.c_uint64),
                ("rows", C.c_uint64), ("row_stride", C.c_uint64)]


def _np_dtype(dtype: str):
    try:
        return _DT[dtype]
    except KeyError:
        raise ValueError(f"oracle dtype must be one of {sorted(_DT)}, not {dtype!r}") from None


def _ptrs(arrs):
    arr = (C.c_void_p * max(1, len(arrs)))()
    for i, a in enumerate(arrs):
        arr[i] = a.ctypes.data if a.size else None
    return arr


def _u64(xs):
    xs = [int(x) for x in xs]
    return (C.c_uint64 * max(1, len(xs)))(*xs)


def _inputs(ins, dtype):
    code, npdt = _np_dtype(dtype)
    out = []
    for a in ins:
        a = np.ascontiguousarray(a)
        if a.dtype != npdt:
            raise TypeError(f"oracle input for {dtype} must be {npdt.__name__}, got {a.dtype}")
        out.append(a)
    return code, npdt, out


def _reducible(dtype):
    if dtype == "fp8":
        raise ValueError("1-byte (fp8) elements are only moved, never reduced")


def f16_to_f32(h) -> np.ndarray:
    """IEEE binary16 bit patterns -> fp32 values (numpy's float16 view; exact)."""
    return np.ascontiguousarray(h, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_to_f32(h) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact: a bf16 is the top half of an fp32)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


class Oracle:
    """The oracle functions bound to one build of ``oracle.c`` (the committed
    build, or a deliberately mutated copy used to show that the pins catch
    mistakes)."""

    def __init__(self, path: str):
        L = C.CDLL(path)
        vp, u64p = C.c_void_p, C.POINTER(C.c_uint64)
        L.orc_f32_to_bf16_n.argtypes = [C.c_void_p, C.c_void_p, C.c_uint64]
        L.orc_f32_to_bf16_n.restype = None
        L.orc_f32_to_f16_n.argtypes = [C.c_void_p, C.c_void_p, C.c_uint64]
        L.orc_f32_to_f16_n.restype = None
        L.orc_reducescatter_op.argtypes = [C.c_int, C.c_int, C.c_int, C.POINTER(vp), u64p, C.POINTER(vp)]
        L.orc_reducescatter_op.restype = None
        L.orc_allreduce_op.argtypes = [C.c_int, C.c_int, C.c_int, C.POINTER(vp), C.c_uint64, C.POINTER(vp)]
        L.orc_allreduce_op.restype = None
        for name in ("orc_allgather", "orc_reducescatter", "orc_alltoall"):
            getattr(L, name).argtypes = [C.c_int, C.c_int, C.POINTER(vp), u64p, C.POINTER(vp)]
            getattr(L, name).restype = None
        L.orc_allreduce.argtypes = [C.c_int, C.c_int, C.POINTER(vp), C.c_uint64, C.POINTER(vp)]
        L.orc_allreduce.restype = None
        L.orc_ulysses.argtypes = [C.c_int, C.c_int, C.POINTER(vp), C.c_uint64, C.c_uint64,
                                  C.c_uint64, C.POINTER(vp)]
        L.orc_ulysses.restype = None
        L.orc_collective.argtypes = [C.c_int, C.c_int, C.c_int,
                                     C.POINTER(C.c_int), C.POINTER(_Part), C.POINTER(vp),
                                     C.POINTER(C.c_int), C.POINTER(_Part), C.POINTER(vp)]
        L.orc_collective.restype = C.c_int
        self.lib = L
        self.path = path

    # ------------------------------------------------------------- rounding

    def f32_to_bf16(self, x) -> np.ndarray:
        """fp32 values -> bf16 bit patterns, IEEE round-to-nearest-even."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        y = np.empty(x.size, dtype=np.uint16)
        if x.size:
            self.lib.orc_f32_to_bf16_n(x.ctypes.data, y.ctypes.data, x.size)
        return y

    def f32_to_f16(self, x) -> np.ndarray:
        """fp32 values -> IEEE binary16 bit patterns, round-to-nearest-even."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        y = np.empty(x.size, dtype=np.uint16)
        if x.size:
            self.lib.orc_f32_to_f16_n(x.ctypes.data, y.ctypes.data, x.size)
        return y

    # ---------------------------------------------------------- collectives

    def allgather(self, ins, dtype: str):
        """AllGather(V): every rank receives every input, in rank order (Figure 4)."""
        code, npdt, ins = _inputs(ins, dtype)
        R = len(ins)
        n = [a.size for a in ins]
        outs = [np.empty(sum(n), dtype=npdt) for _ in range(R)]
        self.lib.orc_allgather(R, code, _ptrs(ins), _u64(n), _ptrs(outs))
        return outs

    def reducescatter(self, ins, lens, dtype: str, op: str = "sum"):
        """ReduceScatter(V): rank k receives the rank-ordered sum (or max) of partition k (Figure 4)."""
        code, npdt, ins = _inputs(ins, dtype)
        _reducible(dtype)
        R = len(ins)
        lens = [int(x) for x in lens]
        if len(lens) != R or any(a.size != sum(lens) for a in ins):
            raise ValueError("reducescatter: each input must hold sum(lens) elements, R = len(lens)")
        outs = [np.empty(lens[k], dtype=npdt) for k in range(R)]
        if op == "sum":
            self.lib.orc_reducescatter(R, code, _ptrs(ins), _u64(lens), _ptrs(outs))
        else:
            self.lib.orc_reducescatter_op(R, code, _OPS[op], _ptrs(ins), _u64(lens), _ptrs(outs))
        return outs

    def allreduce(self, ins, dtype: str, op: str = "sum"):
        """AllReduce: every rank receives the rank-ordered elementwise sum (or max) (direct definition)."""
        code, npdt, ins = _inputs(ins, dtype)
        _reducible(dtype)
        R = len(ins)
        count = ins[0].size
        if any(a.size != count for a in ins):
            raise ValueError("allreduce: inputs must have equal sizes")
        outs = [np.empty(count, dtype=npdt) for _ in range(R)]
        if op == "sum":
            self.lib.orc_allreduce(R, code, _ptrs(ins), count, _ptrs(outs))
        else:
            self.lib.orc_allreduce_op(R, code, _OPS[op], _ptrs(ins), count, _ptrs(outs))
        return outs

    def alltoall(self, ins, lens_matrix, dtype: str):
        """AllToAll(V): rank j receives partition j of every source, in source order (Figure 4).

        ``lens_matrix[r][j]`` is the length of source r's partition for destination j.
        """
        code, npdt, ins = _inputs(ins, dtype)
        R = len(ins)
        m = [[int(x) for x in row] for row in lens_matrix]
        if len(m) != R or any(len(row) != R for row in m):
            raise ValueError("alltoall: lens_matrix must be R x R")
        if any(ins[r].size != sum(m[r]) for r in range(R)):
            raise ValueError("alltoall: input r must hold sum(lens_matrix[r]) elements")
        outs = [np.empty(sum(m[r][j] for r in range(R)), dtype=npdt) for j in range(R)]
        flat = [m[r][j] for r in range(R) for j in range(R)]
        self.lib.orc_alltoall(R, code, _ptrs(ins), _u64(flat), _ptrs(outs))
        return outs

    def ulysses_a2a(self, ins, S: int, H: int, D: int, dtype: str):
        """Sequence -> head re-partition: rank r's [S, H, D] shard; rank j gets heads j*H/R.. of all."""
        code, npdt, ins = _inputs(ins, dtype)
        R = len(ins)
        if H % R:
            raise ValueError("ulysses_a2a: H must be a multiple of R")
        if any(a.size != S * H * D for a in ins):
            raise ValueError("ulysses_a2a: each input must hold S*H*D elements")
        outs = [np.empty(R * S * (H // R) * D, dtype=npdt) for _ in range(R)]
        self.lib.orc_ulysses(R, code, _ptrs(ins), S, H, D, _ptrs(outs))
        return outs

    def collective(self, op: str, dtype: str, in_layout, out_layout, ins, out_sizes):
        """Any collective given as a layout pair (abstract: input layout, output layout, op).

        ``in_layout[r]`` / ``out_layout[r]`` list rank r's parts, each a tuple
        ``(name, offset, len)`` or ``(name, offset, len, rows, row_stride)`` in elements.
        ``out_sizes[r]`` is the element count of rank r's output buffer, which starts
        zero-filled (elements no part names stay zero).
        """
        code, npdt, ins = _inputs(ins, dtype)
        R = len(ins)
        opc = _OPS[op]

        def flat(layout):
            if len(layout) != R:
                raise ValueError("layout must list parts for every rank")
            counts = (C.c_int * R)(*[len(parts) for parts in layout])
            items = []
            for parts in layout:
                for p in parts:
                    p = tuple(int(v) for v in p)
                    if len(p) == 3:
                        p = p + (1, p[2])
                    items.append(_Part(*p))
            arr = (_Part * max(1, len(items)))(*items)
            return counts, arr

        # every part inside its buffer (the C code takes bare pointers)
        for layout, sizes in ((in_layout, [a.size for a in ins]), (out_layout, [int(s) for s in out_sizes])):
            for parts, size in zip(layout, sizes):
                for p in parts:
                    p = tuple(int(v) for v in p)
                    rows, stride = (p[3], p[4]) if len(p) == 5 else (1, p[2])
                    if p[2] and p[1] + (rows - 1) * stride + p[2] > size:
                        raise ValueError("a layout part lies outside its buffer")
        nin, pin = flat(in_layout)
        nout, pout = flat(out_layout)
        outs = [np.zeros(int(s), dtype=npdt) for s in out_sizes]
        rc = self.lib.orc_collective(R, opc, code, nin, pin, _ptrs(ins), nout, pout, _ptrs(outs))
        if rc != 0:
            raise ValueError("layout pair does not name a valid collective")
        return outs


_default = None


def default() -> Oracle:
    """The oracle built from ``oracle.c`` as committed (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def f32_to_bf16(x):
    return default().f32_to_bf16(x)


def f32_to_f16(x):
    return default().f32_to_f16(x)


def allgather(ins, dtype):
    return default().allgather(ins, dtype)


def reducescatter(ins, lens, dtype, op="sum"):
    return default().reducescatter(ins, lens, dtype, op)


def allreduce(ins, dtype, op="sum"):
    return default().allreduce(ins, dtype, op)


def alltoall(ins, lens_matrix, dtype):
    return default().alltoall(ins, lens_matrix, dtype)


def ulysses_a2a(ins, S, H, D, dtype):
    return default().ulysses_a2a(ins, S, H, D, dtype)


def collective(op, dtype, in_layout, out_layout, ins, out_sizes):
    return default().collective(op, dtype, in_layout, out_layout, ins, out_sizes)
