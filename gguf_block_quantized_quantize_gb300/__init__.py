"""GB300-native GGUF block-quantized matmul: thin Python binding of libgguf_gb300.

Each function has the name of the C-ABI entry point it calls and only
marshals arguments (torch CUDA tensors -> device pointers, the current CUDA
stream, workspace allocation through torch's caching allocator).  Every step
of the computation runs in the library's CUDA kernels; there is no fallback:
if the library is missing or the device is not a CUDA GPU, the calls raise.

Packed weights and q8_1 activations are ``torch.uint8`` tensors of shape
``[rows, row_size]``.
"""
from __future__ import annotations

import ctypes
import os

import torch

F32, F16, Q4_0, Q8_0, Q8_1, Q4_K, Q5_K, Q6_K, BF16, MXFP4 = 0, 1, 2, 8, 9, 12, 13, 14, 30, 39
GATE_UP_SWIGLU, DOWN_WEIGHTED_SUM, PLAIN = 0, 1, 2
Q8_1_BYTES = 36   # one q8_1 block: fp16 d, fp16 s, 32 int8 quants (a q8_1 row is k / 32 blocks)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgguf_gb300.so")

_DTYPE_OF = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
_TYPE_OF = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED_TYPE", 3: "SHAPE", 4: "ALIGNMENT", 5: "WORKSPACE", 6: "CUDA",
           7: "DEVICE"}


class GgufError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


MAX_SEGMENTS = 8


class Segment(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("n", ctypes.c_int64), ("y", ctypes.c_void_p), ("ldy", ctypes.c_int64)]


class MmJob(ctypes.Structure):
    _fields_ = [("segs", ctypes.POINTER(Segment)), ("nseg", ctypes.c_int), ("xq", ctypes.c_void_p),
                ("m", ctypes.c_int64)]


class MmJobTyped(ctypes.Structure):
    _fields_ = [("wt", ctypes.c_int), ("k", ctypes.c_int64), ("segs", ctypes.POINTER(Segment)), ("nseg", ctypes.c_int),
                ("xq", ctypes.c_void_p), ("m", ctypes.c_int64)]


MAX_BATCH_JOBS = 8


class MoeArgs(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("wt", ctypes.c_int), ("n_experts", ctypes.c_int64),
                ("expert_stride", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("xt", ctypes.c_int), ("n_tokens", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("ids", ctypes.c_void_p), ("top_k", ctypes.c_int64),
                ("route_w", ctypes.c_void_p), ("mode", ctypes.c_int), ("y", ctypes.c_void_p),
                ("yt", ctypes.c_int), ("dev_status", ctypes.c_void_p)]


class MoeFfnArgs(ctypes.Structure):
    _fields_ = [("w_gate_up", ctypes.c_void_p), ("gate_up_type", ctypes.c_int), ("gate_up_stride", ctypes.c_int64),
                ("w_down", ctypes.c_void_p), ("down_type", ctypes.c_int), ("down_stride", ctypes.c_int64),
                ("n_experts", ctypes.c_int64), ("hidden", ctypes.c_int64), ("inter", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("xt", ctypes.c_int), ("n_tokens", ctypes.c_int64), ("ldx", ctypes.c_int64),
                ("ids", ctypes.c_void_p), ("top_k", ctypes.c_int64), ("route_w", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("yt", ctypes.c_int), ("dev_status", ctypes.c_void_p)]


# name -> (restype, argtypes); the exported C-ABI of include/gguf_gb300.h
_i, _i64, _p, _sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
SIGNATURES = {
    "gguf_last_error": (ctypes.c_char_p, []),
    "gguf_type_block_elems": (_i64, [_i]),
    "gguf_type_block_bytes": (_i64, [_i]),
    "gguf_row_size": (_i64, [_i, _i64]),
    "gguf_quantize_q8_1": (_i, [_p, _i, _i64, _i64, _i64, _p, _p]),
    "gguf_dequantize": (_i, [_p, _i, _i64, _i64, _p, _i, _p]),
    "gguf_copy_async": (_i, [_p, _p, _i64, _p]),
    "gguf_mul_mat_batch_typed": (_i, [ctypes.POINTER(MmJobTyped), _i, _i, _p]),
    "gguf_get_rows": (_i, [_p, _i, _i64, _i64, _p, _i64, _p, _i, _p]),
    "gguf_mul_mat_ws_size": (_sz, [_i, _i64, _i64, _i, _i64, _i]),
    "gguf_mul_mat": (_i, [_p, _i, _i64, _i64, _p, _i, _i64, _i64, _p, _i, _i64, _p, _sz, _p]),
    "gguf_mul_mat_noalloc": (_i, [_p, _i, _i64, _i64, _p, _i, _i64, _i64, _p, _i, _i64, _p]),
    "gguf_mul_mat_segments_ws_size": (_sz, [_i, ctypes.POINTER(Segment), _i, _i64, _i, _i64, _i]),
    "gguf_mul_mat_segments": (_i, [_i, ctypes.POINTER(Segment), _i, _i64, _p, _i, _i64, _i64, _i, _p, _sz, _p]),
    "gguf_mul_mat_batch": (_i, [_i, _i64, ctypes.POINTER(MmJob), _i, _i, _p]),
    "gguf_mul_mat_id_ws_size": (_sz, [ctypes.POINTER(MoeArgs)]),
    "gguf_mul_mat_id": (_i, [ctypes.POINTER(MoeArgs), _p, _sz, _p]),
    "gguf_moe_ffn_ws_size": (_sz, [ctypes.POINTER(MoeFfnArgs)]),
    "gguf_moe_ffn": (_i, [ctypes.POINTER(MoeFfnArgs), _p, _sz, _p]),
    "gguf_debug_block_dots": (_i, [_p, _i, _i64, _i64, _p, _i64, _p, _p]),
    "gguf_set_option": (_i, [ctypes.c_char_p, _i64]),
    "gguf_get_option": (_i64, [ctypes.c_char_p]),
    "gguf_device_errors": (_i, [ctypes.POINTER(ctypes.c_int32), _i, _p]),
    "gguf_device_errors_async": (_i, [_p, _i, _p]),
}

_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgguf_gb300.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libgguf_gb300.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(st: int):
    if st != 0:
        raise GgufError(st, load_library().gguf_last_error().decode())


# the current stream's raw handle without building a Stream object (the
# public call is the fallback)
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream():
    if _RAW_STREAM is not None:
        return _RAW_STREAM(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _lib_fast():
    return _lib if _lib is not None else load_library()


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("gguf: tensors must live on a CUDA device")
    return t.data_ptr()


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def gguf_row_size(t: int, k: int) -> int:
    return int(load_library().gguf_row_size(t, k))


def gguf_set_option(key: str, value: int):
    _check(load_library().gguf_set_option(key.encode(), int(value)))


def gguf_get_option(key: str) -> int:
    return int(load_library().gguf_get_option(key.encode()))


def _check_x_rows(x: torch.Tensor, xt: int, k: int, what: str):
    """The C ABI reads x as rows of k values (or q8_1 bytes) with a row stride:
    the values of a row must be adjacent, and q8_1 rows packed back to back."""
    if x.dim() != 2:
        raise ValueError(f"{what}: x must be a 2-D tensor")
    if xt == Q8_1:
        if x.shape[0] > 1 and x.stride(0) != k // 32 * Q8_1_BYTES or x.shape[1] > 1 and x.stride(1) != 1:
            raise ValueError(f"{what}: q8_1 rows of x must be contiguous")
    elif x.shape[1] > 1 and x.stride(1) != 1:
        raise ValueError(f"{what}: the values of a row of x must be contiguous (stride(1) == 1)")


def gguf_quantize_q8_1(x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """x [m, k] (fp32 / bf16 / fp16, rows may be strided) -> q8_1 bytes [m, k/32*36]."""
    m, k = x.shape
    if x.stride(1) != 1:
        raise ValueError("gguf_quantize_q8_1: rows must be contiguous")
    if out is None:
        out = torch.empty((m, max(gguf_row_size(Q8_1, k), 0)), dtype=torch.uint8, device=x.device)
    _check(_lib_fast().gguf_quantize_q8_1(_ptr(x), _TYPE_OF[x.dtype], m, k, x.stride(0), _ptr(out), _stream()))
    return out


def gguf_copy(dst: torch.Tensor, src: torch.Tensor) -> torch.Tensor:
    """dst <- src on the current stream through gguf_copy_async (a copy on the
    SMs): each tensor contiguous and on the GPU or in pinned host memory, both
    the same number of bytes."""
    for t, what in ((dst, "dst"), (src, "src")):
        if not t.is_contiguous():
            raise ValueError(f"gguf_copy: {what} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"gguf_copy: {what} must be a CUDA tensor or pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("gguf_copy: dst and src differ in size")
    _check(_lib_fast().gguf_copy_async(dst.data_ptr(), src.data_ptr(), nbytes, _stream()))
    return dst


def gguf_dequantize(w: torch.Tensor, wt: int, rows: int, k: int, out_dtype=torch.float32,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    if out is None:
        out = torch.empty((rows, k), dtype=out_dtype, device=w.device)
    _check(load_library().gguf_dequantize(_ptr(w), wt, rows, k, _ptr(out), _TYPE_OF[out.dtype], _stream()))
    return out


def gguf_get_rows(table: torch.Tensor, tt: int, rows: int, k: int, ids: torch.Tensor, out_dtype=torch.float32,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    n = ids.numel()
    if out is None:
        out = torch.empty((n, k), dtype=out_dtype, device=ids.device)
    _check(load_library().gguf_get_rows(_ptr(table), tt, rows, k, _ptr(ids), n, _ptr(out), _TYPE_OF[out.dtype],
                                        _stream()))
    return out


def gguf_mul_mat_ws_size(wt: int, n: int, k: int, xt: int, m: int, yt: int = BF16) -> int:
    return int(load_library().gguf_mul_mat_ws_size(wt, n, k, xt, m, yt))


def gguf_mul_mat(w: torch.Tensor, wt: int, n: int, k: int, x: torch.Tensor, xt: int | None = None,
                 m: int | None = None, out: torch.Tensor | None = None, out_dtype=None,
                 ws: torch.Tensor | None = None) -> torch.Tensor:
    """y[m, n] = x[m, k] @ W[n, k]^T.  ``x`` is a float tensor, or q8_1 bytes
    with ``xt=Q8_1`` (then ``m`` = rows of x).  ``out`` may be a column slice of
    a wider row-major tensor (its row stride becomes ldy)."""
    if xt is None:
        xt = _TYPE_OF[x.dtype]
    if m is None:
        m = x.shape[0]
    _check_x_rows(x, xt, k, "gguf_mul_mat")
    ldx = x.stride(0) if xt != Q8_1 else k // 32 * Q8_1_BYTES
    if out is None:
        if out_dtype is None:
            out_dtype = x.dtype if xt != Q8_1 else torch.float32
        out = torch.empty((m, n), dtype=out_dtype, device=x.device)
    if out.stride(1) != 1:
        raise ValueError("gguf_mul_mat: output rows must be contiguous")
    yt = _TYPE_OF[out.dtype]
    if ws is None:   # a caller's workspace is checked against the need by the library
        ws = _workspace(gguf_mul_mat_ws_size(wt, n, k, xt, m, yt), x.device)
    _check(_lib_fast().gguf_mul_mat(_ptr(w), wt, n, k, _ptr(x), xt, m, ldx, _ptr(out), yt, out.stride(0), _ptr(ws),
                                    0 if ws is None else ws.numel(), _stream()))
    return out


def gguf_mul_mat_segments(wt: int, k: int, x: torch.Tensor, segments, xt: int | None = None, m: int | None = None,
                          ws: torch.Tensor | None = None):
    """y_s = x @ W_s^T for each (w, n, out) in ``segments``, with x quantized once
    (one MMVQ launch for all segments when m is small).  ``out`` tensors must
    have contiguous rows and share one dtype; they are returned."""
    if xt is None:
        xt = _TYPE_OF[x.dtype]
    if m is None:
        m = x.shape[0]
    _check_x_rows(x, xt, k, "gguf_mul_mat_segments")
    ldx = x.stride(0) if xt != Q8_1 else k // 32 * Q8_1_BYTES
    outs = [o for (_, _, o) in segments]
    yt = _TYPE_OF[outs[0].dtype]
    for o in outs:
        if o.stride(1) != 1 or _TYPE_OF[o.dtype] != yt:
            raise ValueError("gguf_mul_mat_segments: outputs need contiguous rows and one dtype")
    arr = (Segment * len(segments))(*[Segment(_ptr(w), n, _ptr(o), o.stride(0)) for (w, n, o) in segments])
    lib = _lib_fast()
    if ws is None:   # a caller's workspace is checked against the need by the library
        ws = _workspace(int(lib.gguf_mul_mat_segments_ws_size(wt, arr, len(segments), k, xt, m, yt)), x.device)
    _check(lib.gguf_mul_mat_segments(wt, arr, len(segments), k, _ptr(x), xt, m, ldx, yt, _ptr(ws),
                                     0 if ws is None else ws.numel(), _stream()))
    return outs


def gguf_mul_mat_batch(wt: int, k: int, jobs):
    """Decode-sized products on q8_1 rows, one chained launch per job:
    ``jobs`` is a list of (xq [m, row bytes] uint8, [(w, n, out), ...]).  The
    outputs share one dtype; they are returned per job."""
    arrs, cjobs, outs = [], [], []
    yt = None
    for xq, segs in jobs:
        if xq.dim() != 2 or (xq.shape[0] > 1 and xq.stride(0) != k // 32 * Q8_1_BYTES):
            raise ValueError("gguf_mul_mat_batch: q8_1 rows of xq must be contiguous")
        for (_, _, o) in segs:
            t = _TYPE_OF[o.dtype]
            if o.stride(1) != 1 or (yt is not None and t != yt):
                raise ValueError("gguf_mul_mat_batch: outputs need contiguous rows and one dtype")
            yt = t
        arr = (Segment * len(segs))(*[Segment(_ptr(w), n, _ptr(o), o.stride(0)) for (w, n, o) in segs])
        arrs.append(arr)
        cjobs.append(MmJob(arr, len(segs), _ptr(xq), xq.shape[0]))
        outs.append([o for (_, _, o) in segs])
    if not cjobs:
        return outs
    carr = (MmJob * len(cjobs))(*cjobs)
    _check(_lib_fast().gguf_mul_mat_batch(wt, k, carr, len(cjobs), yt, _stream()))
    return outs


def _typed_jobs(jobs, what):
    """ctypes typed jobs of [(wt, k, xq, [(w, n, out), ...]), ...]: the arrays
    to keep alive, the jobs, the outputs per job and the one output type."""
    keep, cjobs, outs, yt = [], [], [], None
    for wt, k, xq, segs in jobs:
        if xq.dim() != 2 or (xq.shape[0] > 1 and xq.stride(0) != k // 32 * Q8_1_BYTES):
            raise ValueError(f"{what}: q8_1 rows of xq must be contiguous")
        for (_, _, o) in segs:
            t = _TYPE_OF[o.dtype]
            if o.stride(1) != 1 or (yt is not None and t != yt):
                raise ValueError(f"{what}: outputs need contiguous rows and one dtype")
            yt = t
        arr = (Segment * len(segs))(*[Segment(_ptr(w), n, _ptr(o), o.stride(0)) for (w, n, o) in segs])
        keep.append((xq, segs, arr))
        cjobs.append(MmJobTyped(wt, k, arr, len(segs), _ptr(xq), xq.shape[0]))
        outs.append([o for (_, _, o) in segs])
    return keep, cjobs, outs, yt


def gguf_mul_mat_batch_typed(jobs):
    """gguf_mul_mat_batch with the weight type and K per job: ``jobs`` is a
    list of (wt, k, xq [m, row bytes] uint8, [(w, n, out), ...]).  The outputs
    share one dtype; they are returned per job."""
    keep, cjobs, outs, yt = _typed_jobs(jobs, "gguf_mul_mat_batch_typed")
    if not cjobs:
        return outs
    carr = (MmJobTyped * len(cjobs))(*cjobs)
    _check(_lib_fast().gguf_mul_mat_batch_typed(carr, len(cjobs), yt, _stream()))
    del keep
    return outs


class PreparedBatch:
    """The arguments of one gguf_mul_mat_batch call marshalled once (the
    tensors are referenced, not copied): ``run()`` issues the call on the
    current stream with no per-call argument building, as an engine that
    replays the same decode step does.  Same ``jobs`` as gguf_mul_mat_batch."""

    def __init__(self, wt: int, k: int, jobs):
        self._keep, cjobs, yt = [], [], None
        for xq, segs in jobs:
            if xq.dim() != 2 or (xq.shape[0] > 1 and xq.stride(0) != k // 32 * Q8_1_BYTES):
                raise ValueError("PreparedBatch: q8_1 rows of xq must be contiguous")
            for (_, _, o) in segs:
                t = _TYPE_OF[o.dtype]
                if o.stride(1) != 1 or (yt is not None and t != yt):
                    raise ValueError("PreparedBatch: outputs need contiguous rows and one dtype")
                yt = t
            arr = (Segment * len(segs))(*[Segment(_ptr(w), n, _ptr(o), o.stride(0)) for (w, n, o) in segs])
            self._keep.append((xq, segs, arr))
            cjobs.append(MmJob(arr, len(segs), _ptr(xq), xq.shape[0]))
        self._args = (wt, k, (MmJob * len(cjobs))(*cjobs), len(cjobs), yt)

    def run(self):
        _check(_lib_fast().gguf_mul_mat_batch(*self._args, _stream()))


def gguf_mul_mat_noalloc(w: torch.Tensor, wt: int, n: int, k: int, x: torch.Tensor,
                         out: torch.Tensor | None = None, out_dtype=None) -> torch.Tensor:
    """y[m, n] = x[m, k] @ W[n, k]^T for m <= 8, k <= 16384, with the q8_1
    scratch in the library's fixed device array (no workspace, no allocation
    inside the call; calls that overlap on one device race on the scratch)."""
    xt = _TYPE_OF[x.dtype]
    m = x.shape[0]
    _check_x_rows(x, xt, k, "gguf_mul_mat_noalloc")
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype or x.dtype, device=x.device)
    if out.stride(1) != 1:
        raise ValueError("gguf_mul_mat_noalloc: output rows must be contiguous")
    _check(load_library().gguf_mul_mat_noalloc(_ptr(w), wt, n, k, _ptr(x), xt, m, x.stride(0), _ptr(out),
                                               _TYPE_OF[out.dtype], out.stride(0), _stream()))
    return out


def moe_args(w, wt, n_experts, expert_stride, n, k, x, xt, n_tokens, ldx, ids, top_k, route_w, mode, y, yt,
             dev_status=None) -> MoeArgs:
    return MoeArgs(w.data_ptr(), wt, n_experts, expert_stride, n, k, x.data_ptr(), xt, n_tokens, ldx,
                   ids.data_ptr(), top_k, 0 if route_w is None else route_w.data_ptr(), mode, y.data_ptr(), yt,
                   0 if dev_status is None else dev_status.data_ptr())


def gguf_mul_mat_id_ws_size(args: MoeArgs) -> int:
    return int(load_library().gguf_mul_mat_id_ws_size(ctypes.byref(args)))


def gguf_mul_mat_id(w: torch.Tensor, wt: int, n_experts: int, expert_stride: int, n: int, k: int, x: torch.Tensor,
                    ids: torch.Tensor, mode: int, route_w: torch.Tensor | None = None, xt: int | None = None,
                    out_type: int | None = None, out: torch.Tensor | None = None,
                    dev_status: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """MoE expert product (see include/gguf_gb300.h for the three modes)."""
    n_tokens, top_k = ids.shape
    if xt is None:
        xt = _TYPE_OF[x.dtype]
    _check_x_rows(x, xt, k, "gguf_mul_mat_id")
    ldx = x.stride(0) if xt != Q8_1 else gguf_row_size(Q8_1, k)
    if out is None:
        if mode == GATE_UP_SWIGLU:
            yt = BF16 if out_type is None else out_type
            i_dim = n // 2
            if yt in (BF16, F16):
                out = torch.empty((n_tokens * top_k, i_dim), dtype=_DTYPE_OF[yt], device=x.device)
            else:
                out = torch.empty((n_tokens * top_k, gguf_row_size(Q8_1, i_dim)), dtype=torch.uint8, device=x.device)
        else:
            yt = BF16 if out_type is None else out_type
            rows = n_tokens * top_k if mode == PLAIN else n_tokens
            out = torch.empty((rows, n), dtype=_DTYPE_OF[yt], device=x.device)
    else:
        yt = out_type if out_type is not None else (Q8_1 if out.dtype == torch.uint8 else _TYPE_OF[out.dtype])
    args = moe_args(w, wt, n_experts, expert_stride, n, k, x, xt, n_tokens, ldx, ids, top_k, route_w, mode, out,
                    yt, dev_status)
    need = gguf_mul_mat_id_ws_size(args)
    if ws is None:
        ws = _workspace(need, x.device)
    _check(load_library().gguf_mul_mat_id(ctypes.byref(args), _ptr(ws), 0 if ws is None else ws.numel(), _stream()))
    return out


def moe_ffn_args(w_gate_up, gate_up_type, gate_up_stride, w_down, down_type, down_stride, n_experts, hidden, inter,
                 x, xt, ids, top_k, route_w, y, yt, dev_status=None) -> MoeFfnArgs:
    return MoeFfnArgs(w_gate_up.data_ptr(), gate_up_type, gate_up_stride, w_down.data_ptr(), down_type, down_stride,
                      n_experts, hidden, inter, x.data_ptr(), xt, ids.shape[0], x.stride(0) if xt != Q8_1 else 0,
                      ids.data_ptr(), top_k, 0 if route_w is None else route_w.data_ptr(), y.data_ptr(), yt,
                      0 if dev_status is None else dev_status.data_ptr())


def gguf_moe_ffn_ws_size(args: MoeFfnArgs) -> int:
    return int(load_library().gguf_moe_ffn_ws_size(ctypes.byref(args)))


def gguf_moe_ffn(w_gate_up: torch.Tensor, gate_up_type: int, gate_up_stride: int, w_down: torch.Tensor,
                 down_type: int, down_stride: int, n_experts: int, hidden: int, inter: int, x: torch.Tensor,
                 ids: torch.Tensor, route_w: torch.Tensor | None, out: torch.Tensor | None = None,
                 dev_status: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """The whole MoE expert block: y = sum_k w_k * down_e(silu(gate_e x) * up_e x)."""
    n_tokens, top_k = ids.shape
    xt = _TYPE_OF[x.dtype] if x.dtype != torch.uint8 else Q8_1
    _check_x_rows(x, xt, hidden, "gguf_moe_ffn")
    if out is None:
        out = torch.empty((n_tokens, hidden), dtype=x.dtype if xt != Q8_1 else torch.bfloat16, device=x.device)
    args = moe_ffn_args(w_gate_up, gate_up_type, gate_up_stride, w_down, down_type, down_stride, n_experts, hidden,
                        inter, x, xt, ids, top_k, route_w, out, _TYPE_OF[out.dtype], dev_status)
    need = gguf_moe_ffn_ws_size(args)
    if ws is None:
        ws = _workspace(need, x.device)
    _check(load_library().gguf_moe_ffn(ctypes.byref(args), _ptr(ws), 0 if ws is None else ws.numel(), _stream()))
    return out


def gguf_device_errors(clear: bool = True) -> int:
    """Error word of the tensor-core kernels after the current stream's work;
    raises GgufError (status DEVICE) when a kernel gave up a bounded wait."""
    v = ctypes.c_int32(0)
    _check(load_library().gguf_device_errors(ctypes.byref(v), 1 if clear else 0, _stream()))
    return int(v.value)


def gguf_device_errors_async(out: torch.Tensor, clear: bool = True) -> torch.Tensor:
    """Stream-ordered copy of the error word into the int32 device tensor ``out``."""
    if out.dtype != torch.int32 or out.numel() < 1:
        raise ValueError("gguf_device_errors_async: out must be an int32 tensor with one element")
    _check(load_library().gguf_device_errors_async(_ptr(out), 1 if clear else 0, _stream()))
    return out


def gguf_debug_block_dots(w: torch.Tensor, wt: int, n: int, k: int, xq: torch.Tensor, m: int) -> torch.Tensor:
    sub = 16 if wt == Q6_K else 32
    out = torch.empty((m, n, k // sub), dtype=torch.int32, device=xq.device)
    _check(load_library().gguf_debug_block_dots(_ptr(w), wt, n, k, _ptr(xq), m, _ptr(out), _stream()))
    return out
