"""NVFP4 block quantization on GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libnvfp4_gb300.so`` (the C ABI in
``include/nvfp4.h``).  It only marshals arguments: torch supplies device
memory and the current stream, and every step of quantization runs in the
library's CUDA kernels.  There is no CPU or eager fallback: if the library is
not built, or no CUDA device is present, calls raise.

Functions (same names as the C ABI):
  nvfp4_quantize(x, ...)   -> dict(codes, scales[, codes_col, scales_col][, gamax])
  nvfp4_dequantize(codes, scales, M, K, ...) -> tensor
  nvfp4_qdq(x, ...)        -> dict(out[, codes, scales][, gamax])
  nvfp4_amax(x, ...)       -> tensor
Calls on CUDA tensors stay on their device.  Calls on CPU tensors (the
host-buffer path) stage their inputs on the current CUDA device and copy the
results back (into the caller's host tensors when given, else into new pinned
ones); they return with their results ready.  Host calls of 256 rows or more
whose rows are independent run in row chunks, with the copies in, the
kernels and the copies out of successive chunks overlapping.  With
``non_blocking=True`` a host call returns once its copies and kernels are
enqueued, so successive calls overlap too (one call's inputs going in while
an earlier call's results come back); nvfp4_synchronize() waits for them.  A
host tensor that a pending call writes is read by later calls only after
that write.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH, build  # noqa: F401  (build is re-exported)

F32, BF16 = 0, 1
BLOCK_1X16, BLOCK_16X16 = 0, 1
RTN, SR, RTN_STD = 0, 1, 2
GAMAX_NONE, GAMAX_TENSOR, GAMAX_ROW, GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN = 0, 1, 2, 3, 4
ERR_NONE, ERR_MAE, ERR_MSE = 0, 1, 2
OK, EINVAL, ECUDA = 0, 1, 2

_NAMES = {
    "block": {"1x16": BLOCK_1X16, "16x16": BLOCK_16X16},
    "rounding": {"rtn": RTN, "sr": SR, "rtn_std": RTN_STD},
    "gamax_mode": {"none": GAMAX_NONE, "tensor": GAMAX_TENSOR, "row": GAMAX_ROW,
                   "tensor_given": GAMAX_TENSOR_GIVEN, "row_given": GAMAX_ROW_GIVEN},
    "err_mode": {"none": ERR_NONE, "mae": ERR_MAE, "mse": ERR_MSE},
    "dtype": {"f32": F32, "bf16": BF16},
}

EXPORTED = ("nvfp4_quantize", "nvfp4_dequantize", "nvfp4_qdq", "nvfp4_amax",
            "nvfp4_global_scales", "nvfp4_probe_divide", "nvfp4_probe_e2m1", "nvfp4_probe_sub_f16", "nvfp4_last_error",
            "nvfp4_abi_version")

_lock = threading.Lock()
_lib = None


class NVFP4Error(RuntimeError):
    """A non-OK status from the library (message from nvfp4_last_error)."""

    def __init__(self, status: int, message: str):
        super().__init__(f"nvfp4 status {status}: {message}")
        self.status = status


def load_library(path: str | None = None):
    """Load the C library (no CUDA call is made).  Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it first with "
                               "nvfp4_block_quantization_quantize_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P, i64, u64, i32, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int,
                                 ctypes.c_float)
        lib.nvfp4_quantize.restype = i32
        lib.nvfp4_quantize.argtypes = [P, i64, i64, i32, i32, i32, P, u64, u64, i64, i32, P, i32,
                                       f32, P, P, P, P, P]
        lib.nvfp4_qdq.restype = i32
        lib.nvfp4_qdq.argtypes = [P, i64, i64, i32, i32, i32, P, u64, u64, i64, i32, P, i32, f32,
                                  P, P, P, P]
        lib.nvfp4_dequantize.restype = i32
        lib.nvfp4_dequantize.argtypes = [P, P, i64, i64, i32, P, f32, P, i32, P]
        lib.nvfp4_amax.restype = i32
        lib.nvfp4_amax.argtypes = [P, i64, i64, i32, P, i32, P, P]
        lib.nvfp4_probe_divide.restype = i32
        lib.nvfp4_probe_divide.argtypes = [P, P, P, i64, P]
        lib.nvfp4_probe_sub_f16.restype = i32
        lib.nvfp4_probe_sub_f16.argtypes = [P, P, P, i64, P]
        lib.nvfp4_global_scales.restype = i32
        lib.nvfp4_global_scales.argtypes = [P, i64, f32, P, P, P]
        lib.nvfp4_probe_e2m1.restype = i32
        lib.nvfp4_probe_e2m1.argtypes = [ctypes.c_uint32, i64, P, P]
        lib.nvfp4_scales_to_mma.restype = i32
        lib.nvfp4_scales_to_mma.argtypes = [P, i64, i64, P, P]
        lib.nvfp4_mm.restype = i32
        lib.nvfp4_mm.argtypes = [P, P, P, P, i64, i64, i64, P, P, f32, P, i32, P]
        lib.nvfp4_last_error.restype = ctypes.c_char_p
        lib.nvfp4_last_error.argtypes = []
        lib.nvfp4_abi_version.restype = i32
        lib.nvfp4_abi_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def _enum(kind: str, v) -> int:
    if isinstance(v, str):
        try:
            return _NAMES[kind][v.lower()]
        except KeyError:
            raise ValueError(f"unknown {kind} {v!r}; expected one of {list(_NAMES[kind])}")
    return int(v)


def _check(lib, rc: int):
    if rc != OK:
        raise NVFP4Error(rc, lib.nvfp4_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _x_dtype(x: torch.Tensor) -> int:
    if x.dtype == torch.float32:
        return F32
    if x.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")


def _device_of(*ts):
    for t in ts:
        if t is not None and t.is_cuda:
            return t.device
    if not torch.cuda.is_available():
        raise RuntimeError("nvfp4: no CUDA device (this library has no CPU path)")
    return torch.device("cuda", torch.cuda.current_device())


def _stage(t, dev):
    if t is None or t.device == dev:
        return t
    if not t.is_cuda:                           # after any pending write of it
        _wait_pending(dev, torch.cuda.current_stream(dev), [t])
    return t.to(dev, non_blocking=True)


def _empty(shape, dtype, dev):
    return torch.empty(shape, dtype=dtype, device=dev)


# ---- host buffers ---------------------------------------------------------------------------
# A call whose tensors live in host memory runs the same kernels on staged
# device copies: inputs (and the residual) are copied to the device, outputs
# are made in device memory and copied back, into the caller's host tensors
# when given, else into new pinned ones.  Host calls return with their
# results ready unless they are non-blocking (below).  (Kernels reading and
# writing mapped pinned memory in place
# over the host link measured 2-2.5x slower than these bulk copies.)
def _host_in(t, dev, name="input"):
    """An input (or the in-place residual) of a host call: a host tensor is
    staged on the call's device; a device tensor must already be there (the
    kernels take its pointer) and is made contiguous (an in-place residual is
    checked to be contiguous before, so it is passed itself)."""
    if t is None:
        return t
    if t.is_cuda:
        if t.device != dev:
            raise ValueError(f"nvfp4: {name} must be on {dev} (got {t.device})")
        return t.contiguous()
    return _stage(t.contiguous(), dev)


def _numel(shape):
    n = 1
    for s in shape:
        n *= int(s)
    return n


def _check_dev(t, name, dtype, numel, dev, at_least=False):
    """A device tensor the kernels read or write through a raw pointer: it must
    be on the call's device, of the expected dtype, contiguous, and hold the
    expected number of elements (at least that many when at_least)."""
    if not t.is_cuda or t.device != dev:
        raise ValueError(f"nvfp4: {name} must be on {dev} (got {t.device})")
    if t.dtype != dtype:
        raise ValueError(f"nvfp4: {name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"nvfp4: {name} must be contiguous")
    if (t.numel() < numel) if at_least else (t.numel() != numel):
        raise ValueError(f"nvfp4: {name} must hold {'at least ' if at_least else ''}{numel} elements "
                         f"(got {t.numel()})")
    return t


def _out_buf(shape, dtype, given, dev, host, name="output"):
    """An output: the given device tensor (checked) or a new device one
    (copied back into a given host tensor by _finish_host); a call on device
    tensors refuses host outputs."""
    if given is not None and given.is_cuda:
        return _check_dev(given, name, dtype, _numel(shape), dev)
    if given is not None and not host:
        raise ValueError("nvfp4: the outputs of a call on device tensors must be device tensors")
    if given is not None and (given.dtype != dtype or given.numel() != _numel(shape)):
        raise ValueError(f"nvfp4: {name} must be {dtype} with {_numel(shape)} elements")
    return _empty(shape, dtype, dev)


def _dev_residual(residual, dev, M=None, K=None):
    """The in-place residual of a call on device tensors: float32 [M,K],
    contiguous, on the call's device (a staged copy would lose the update)."""
    if residual is None:
        return None
    if residual.device != dev:
        raise ValueError("nvfp4: the residual of a call on device tensors must be on x's device")
    if M is None:
        return residual
    return _check_dev(residual, "residual", torch.float32, M * K, dev)


def _host_residual(residual, M, K, dev=None):
    """The residual of a host call: a host float32 tensor of M*K elements
    (staged and copied back), or a device one the kernels update in place,
    which must then be float32 [M,K], contiguous and on the call's device."""
    if residual is None:
        return
    if residual.is_cuda:
        _check_dev(residual, "residual", torch.float32, M * K, dev)
    elif residual.dtype != torch.float32 or residual.numel() != M * K:
        raise ValueError("nvfp4: the residual must be float32 with M*K elements")


def _inputs_ready(stream):
    """Staging copies run on torch's current stream; a call on another stream
    waits for them."""
    if stream is not None:
        torch.cuda.current_stream().synchronize()


def _finish_host(res: dict, given: dict, stream=None) -> dict:
    """End of a host call: results still in device memory are copied into the
    caller's host tensor or a new pinned one, after the call's stream is done;
    then one wait, so everything is ready on return."""
    _sync(stream)
    dev = next(iter(res.values())).device
    _wait_pending(dev, torch.cuda.current_stream(dev), [g for g in given.values() if torch.is_tensor(g) and not g.is_cuda])
    out = {}
    for k, v in res.items():
        g = given.get(k)
        if not v.is_cuda or (g is not None and g.is_cuda):
            out[k] = v
        elif g is not None:
            dst = g if g.shape == v.shape else g.reshape(-1)[:v.numel()].view(v.shape)
            dst.copy_(v, non_blocking=True)
            out[k] = g
        else:
            h = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
            h.copy_(v, non_blocking=True)
            out[k] = h
    torch.cuda.current_stream().synchronize()
    return out


# ---- pipelined host calls ---------------------------------------------------------------------
# A host call whose rows are independent (no columnwise output, no amax over
# the whole tensor, the default stream) runs in row chunks on three streams:
# chunk k+1's inputs go to the device while chunk k's kernels run and chunk
# k-1's results come back, so both directions of the host link carry data at
# once (one direction alone moves ~210 GB/s on this machine, both together
# ~340 GB/s).  Chunks start on multiples of 16 rows (whole 16x16 tiles), and
# each chunk's kernels get row_offset + its first row, so stochastic rounding
# draws the same words and the bytes equal one call's.
_PIPE_CHUNKS = 4
_PIPE_MIN_ROWS = 256
_pipe_lock = threading.Lock()
_pipe_streams = {}
# Non-blocking host calls (non_blocking=True) enqueue the same three streams
# and return at once; their host outputs are written when the copies out
# finish.  _pending[dev] lists (first byte, end byte, event) of host memory
# still being written: a later host call whose input overlaps one waits for
# that event before copying it in.  nvfp4_synchronize() (or any device-wide
# synchronize) makes every result of the device's host calls ready.
_pending = {}


def _row_chunks(M: int):
    """[r0, r1) row ranges: up to _PIPE_CHUNKS, each a multiple of 16 rows
    except the last, covering 0..M."""
    n = max(1, min(_PIPE_CHUNKS, M // 128))
    step = -(-M // n)
    step = -(-step // 16) * 16
    return [(r, min(r + step, M)) for r in range(0, M, step)]


def _pipe_streams_for(dev):
    with _pipe_lock:
        st = _pipe_streams.get(dev)
        if st is None:
            st = tuple(torch.cuda.Stream(device=dev) for _ in range(3))
            _pipe_streams[dev] = st
        return st


def _rows_view(t, M):
    """t as [M, -1] rows when that is a view (contiguous), else None."""
    if t is None:
        return None
    if not t.is_contiguous() or t.numel() % max(M, 1):
        return None
    return t.view(M, -1)


def _host_range(t):
    """[first byte, end byte) of a host tensor's storage."""
    st = t.untyped_storage()
    return st.data_ptr(), st.data_ptr() + st.nbytes()


def _ranges_overlap(a, b) -> bool:
    return a[0] < b[1] and b[0] < a[1]


def _wait_pending(dev, stream, hosts):
    """Make stream wait for the unfinished non-blocking copies out that write
    host memory overlapping any of hosts; finished ones are dropped."""
    with _pipe_lock:
        pend = [p for p in _pending.get(dev, []) if not p[2].query()]
        _pending[dev] = pend
        if not pend:
            return
        for h in hosts:
            r = _host_range(h)
            for lo, hi, ev in pend:
                if _ranges_overlap(r, (lo, hi)):
                    stream.wait_event(ev)


def _add_pending(dev, hosts, ev):
    with _pipe_lock:
        _pending.setdefault(dev, []).extend((*_host_range(h), ev) for h in hosts)


def nvfp4_synchronize(device=None) -> None:
    """Wait until every host call on the device (the current one by default),
    non-blocking ones included, has finished and its results are in host
    memory."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    for st in _pipe_streams_for(dev):
        st.synchronize()
    torch.cuda.current_stream(dev).synchronize()
    with _pipe_lock:
        _pending.pop(dev, None)


def _pipelined(dev, M: int, ins, outs, launch, lib, blocking: bool = True, whole: bool = False, keep=()):
    """ins: (host, device) row-major pairs copied in chunk by chunk; outs:
    (device, host) pairs copied back; launch(r0, r1, stream) enqueues the
    kernels of rows [r0, r1) and returns the library status.  whole: one
    chunk, the tensors copied whole (any shapes).  Returns with everything
    done, or (not blocking) with everything enqueued: the device buffers are
    kept from reuse until the streams pass them, and the host outputs are
    recorded as pending.  keep: device buffers the kernels use besides those."""
    cur = torch.cuda.current_stream(dev)
    s_in, s_cmp, s_out = _pipe_streams_for(dev)
    for st in (s_in, s_cmp, s_out):
        st.wait_stream(cur)
    _wait_pending(dev, s_in, [h for h, _ in ins])
    rc = OK
    for r0, r1 in ([(0, M)] if whole else _row_chunks(M)):
        with torch.cuda.stream(s_in):
            for h, d in ins:
                (d if whole else d[r0:r1]).copy_(h if whole else h[r0:r1], non_blocking=True)
        s_cmp.wait_stream(s_in)
        with torch.cuda.device(dev):
            rc = launch(r0, r1, s_cmp)
        if rc != OK:
            break
        s_out.wait_stream(s_cmp)
        with torch.cuda.stream(s_out):
            for d, h in outs:
                (h if whole else h[r0:r1]).copy_(d if whole else d[r0:r1], non_blocking=True)
    if blocking or rc != OK:
        for st in (s_in, s_cmp, s_out):
            st.synchronize()
        _check(lib, rc)
        return
    for d in [d for _, d in ins] + [d for d, _ in outs] + [d for d in keep if d is not None]:
        for st in (s_in, s_cmp, s_out):
            d.record_stream(st)
    ev = torch.cuda.Event()
    ev.record(s_out)
    _add_pending(dev, [h for _, h in outs], ev)


def _host_out(given, shape, dtype):
    """The host tensor a pipelined call writes: the caller's, else new pinned."""
    if given is not None:
        return given
    return torch.empty(shape, dtype=dtype, pin_memory=True)


def _host_given(t, name, dtype, n):
    """A caller's host output of a pipelined call: None when it cannot be
    written by whole or row-range copies (a device tensor, not contiguous)."""
    if t is None:
        return True
    if t.is_cuda or not t.is_contiguous():
        return False
    if t.dtype != dtype or t.numel() != n:
        raise ValueError(f"nvfp4: {name} must be {dtype} with {n} elements")
    return True


def _gamax_host(gm, gamax, need):
    """Host tensor a computed gamax (tensor / row) is copied into: the
    caller's (its first need values) or a new pinned one."""
    if torch.is_tensor(gamax) and not gamax.is_cuda:
        return gamax.reshape(-1)[:need]
    return torch.empty((need,), dtype=torch.float32, pin_memory=True)


def _sync(stream=None):
    if stream is None:
        torch.cuda.current_stream().synchronize()
    elif isinstance(stream, torch.cuda.Stream):
        stream.synchronize()
    else:
        torch.cuda.synchronize()


def _default_bound(err_mode: int, scale_bound):
    if scale_bound is not None:
        return float(scale_bound)
    return 448.0 if err_mode == ERR_NONE else 256.0


def _gamax_buffer(mode: int, gamax, M: int, dev, host: bool = False):
    """The device buffer the kernels read (GIVEN modes) or write (TENSOR /
    ROW: 1 or M floats, reduced with device atomics).  A device call must pass
    a written gamax as a float32 CUDA tensor on x's device; a host call may
    pass a host tensor, which _finish_host fills from a device buffer."""
    need = 1 if mode in (GAMAX_TENSOR, GAMAX_TENSOR_GIVEN) else max(M, 1)
    if mode in (GAMAX_TENSOR, GAMAX_ROW):
        if gamax is not None:
            if not torch.is_tensor(gamax):
                raise ValueError("nvfp4: a computed gamax is written into a tensor")
            if gamax.is_cuda:
                return _check_dev(gamax, "gamax", torch.float32, need, dev, at_least=True)
            if not host:
                raise ValueError("nvfp4: the gamax of a call on device tensors must be a device tensor")
            if gamax.dtype != torch.float32 or gamax.numel() < need:
                raise ValueError(f"nvfp4: gamax must be float32 with at least {need} elements")
        return _empty((need,), torch.float32, dev)
    if mode in (GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN):
        if gamax is None:
            raise ValueError("a *_given gamax_mode needs gamax")
        if not torch.is_tensor(gamax):
            gamax = torch.tensor([float(gamax)], dtype=torch.float32)
        g = _stage(gamax, dev).to(torch.float32).reshape(-1).contiguous()
        if g.numel() < need:
            raise ValueError(f"nvfp4: gamax must hold at least {need} values")
        return g
    return None


def nvfp4_quantize(x: torch.Tensor, *, block="1x16", rounding="rtn", residual=None, seed: int = 0,
                   step: int = 0, row_offset: int = 0, gamax_mode="none", gamax=None,
                   err_mode="none", scale_bound=None, colwise: bool = False, codes=None,
                   scales=None, codes_col=None, scales_col=None, stream=None,
                   non_blocking: bool = False) -> dict:
    """NVFP4 quantize of a row-major [M,K] float32/bfloat16 tensor (see nvfp4.h).

    ``residual`` (float32 [M,K]) is updated in place.  Output tensors may be
    passed in; otherwise they are allocated with torch on x's device.  A host
    call with ``non_blocking`` returns once its copies and kernels are
    enqueued: its outputs (and the residual) hold the results after
    nvfp4_synchronize(), and its inputs must stay unchanged until then."""
    lib = load_library()
    host = not x.is_cuda
    dev = _device_of(x, residual)
    M, K = x.shape
    blk, rnd = _enum("block", block), _enum("rounding", rounding)
    gm, em = _enum("gamax_mode", gamax_mode), _enum("err_mode", err_mode)
    bound = _default_bound(em, scale_bound)
    given = {"codes": codes, "scales": scales, "codes_col": codes_col, "scales_col": scales_col}
    if host:
        _host_residual(residual, M, K, dev)
        _non_blocking_stream(non_blocking, stream)
        rows = not colwise and M >= _PIPE_MIN_ROWS and gm in (GAMAX_NONE, GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN)
        if stream is None and (rows or non_blocking):
            r = _quantize_pipelined(lib, x, dev, M, K, blk, rnd, residual, seed, step, row_offset, gm,
                                    gamax, em, bound, codes, scales, codes_col, scales_col, colwise,
                                    not non_blocking, not rows)
            if r is not None:
                return r
        _non_blocking_refused(non_blocking)
    xd = _host_in(x, dev) if host else x.contiguous()
    rd = _host_in(residual, dev) if host else _dev_residual(residual, dev, M, K)
    g = _gamax_buffer(gm, gamax, M, dev, host)
    if host and torch.is_tensor(gamax) and not gamax.is_cuda and gm in (GAMAX_TENSOR, GAMAX_ROW):
        given["gamax"] = gamax
    codes = _out_buf((M, K // 2), torch.uint8, codes, dev, host, "codes")
    scales = _out_buf((M, K // 16), torch.uint8, scales, dev, host, "scales")
    if colwise:
        codes_col = _out_buf((K, M // 2), torch.uint8, codes_col, dev, host, "codes_col")
        scales_col = _out_buf((K, M // 16), torch.uint8, scales_col, dev, host, "scales_col")
    if host:
        _inputs_ready(stream)
    with torch.cuda.device(dev):
        rc = lib.nvfp4_quantize(_ptr(xd), M, K, _x_dtype(x), blk, rnd, _ptr(rd), seed, step,
                                row_offset, gm, _ptr(g), em, bound, _ptr(codes), _ptr(scales),
                                _ptr(codes_col), _ptr(scales_col), _stream(stream))
    _check(lib, rc)
    out = {"codes": codes, "scales": scales}
    if colwise:
        out["codes_col"], out["scales_col"] = codes_col, scales_col
    if g is not None:
        out["gamax"] = g
    if host:
        if residual is not None and rd is not residual:
            given["residual"] = residual
            out["residual"] = rd
        out = _finish_host(out, given, stream)
        out.pop("residual", None)
    return out


def _non_blocking_stream(non_blocking, stream):
    if non_blocking and stream is not None:
        raise ValueError("nvfp4: a non-blocking host call runs on the library's own streams (stream=None)")


def _non_blocking_refused(non_blocking):
    if non_blocking:
        raise ValueError("nvfp4: a non-blocking host call takes contiguous host tensors")


def _quantize_pipelined(lib, x, dev, M, K, blk, rnd, residual, seed, step, row_offset, gm, gamax, em, bound,
                        codes, scales, codes_col=None, scales_col=None, colwise=False, blocking=True,
                        whole=False):
    """The host path of nvfp4_quantize through _pipelined: in row chunks, or
    (whole) as one chunk for a call whose rows are not independent; None
    when a host tensor cannot be copied that way (not contiguous, a device
    output)."""
    xh, rh = _rows_view(x, M), _rows_view(residual, M)
    if xh is None or (residual is not None and rh is None):
        return None
    outs_given = [(codes, "codes", M * K // 2), (scales, "scales", M * K // 16)]
    if colwise:
        outs_given += [(codes_col, "codes_col", K * M // 2), (scales_col, "scales_col", K * M // 16)]
    for t, name, n in outs_given:
        if not _host_given(t, name, torch.uint8, n):
            return None
    g = _gamax_buffer(gm, gamax, M, dev, True)
    ch = _host_out(codes, (M, K // 2), torch.uint8)
    sh = _host_out(scales, (M, K // 16), torch.uint8)
    xd = _empty((M, K), x.dtype, dev)
    rd = _empty((M, K), torch.float32, dev) if residual is not None else None
    cd, sd = _empty((M, K // 2), torch.uint8, dev), _empty((M, K // 16), torch.uint8, dev)
    ins = [(xh, xd)] + ([(rh, rd)] if rd is not None else [])
    outs = [(cd, _rows_view(ch, M)), (sd, _rows_view(sh, M))] + ([(rd, rh)] if rd is not None else [])
    ccd = scd = cch = sch = gh = None
    if colwise:
        ccd, scd = _empty((K, M // 2), torch.uint8, dev), _empty((K, M // 16), torch.uint8, dev)
        cch = _host_out(codes_col, (K, M // 2), torch.uint8)
        sch = _host_out(scales_col, (K, M // 16), torch.uint8)
        outs += [(ccd, cch.view(K, M // 2)), (scd, sch.view(K, M // 16))]
    computed = gm in (GAMAX_TENSOR, GAMAX_ROW)
    if computed:
        gh = _gamax_host(gm, gamax, g.numel())
        outs.append((g, gh))

    def launch(r0, r1, st):
        gp = g if (g is None or gm != GAMAX_ROW_GIVEN) else g[r0:]
        return lib.nvfp4_quantize(_ptr(xd[r0]), r1 - r0, K, _x_dtype(x), blk, rnd,
                                  _ptr(None if rd is None else rd[r0]), seed, step, row_offset + r0, gm,
                                  _ptr(gp), em, bound, _ptr(cd[r0]), _ptr(sd[r0]), _ptr(ccd), _ptr(scd),
                                  ctypes.c_void_p(st.cuda_stream))

    _pipelined(dev, M, ins, outs, launch, lib, blocking, whole, keep=(g,))
    out = {"codes": ch, "scales": sh}
    if colwise:
        out["codes_col"], out["scales_col"] = cch, sch
    if computed:
        out["gamax"] = gamax if torch.is_tensor(gamax) and not gamax.is_cuda else gh
    elif g is not None:
        out["gamax"] = g.cpu()
    return out


def _qdq_pipelined(lib, x, dev, M, K, blk, rnd, residual, seed, step, row_offset, gm, gamax, em, bound,
                   out, want_codes, blocking=True, whole=False):
    """The host path of nvfp4_qdq through _pipelined; None as _quantize_pipelined."""
    xh, rh = _rows_view(x, M), _rows_view(residual, M)
    if xh is None or (residual is not None and rh is None):
        return None
    if not _host_given(out, "out", torch.bfloat16, M * K):
        return None
    g = _gamax_buffer(gm, gamax, M, dev, True)
    oh = _host_out(out, (M, K), torch.bfloat16)
    xd = _empty((M, K), x.dtype, dev)
    rd = _empty((M, K), torch.float32, dev) if residual is not None else None
    od = _empty((M, K), torch.bfloat16, dev)
    cd = _empty((M, K // 2), torch.uint8, dev) if want_codes else None
    sd = _empty((M, K // 16), torch.uint8, dev) if want_codes else None
    ch = _host_out(None, (M, K // 2), torch.uint8) if want_codes else None
    sh = _host_out(None, (M, K // 16), torch.uint8) if want_codes else None
    ins = [(xh, xd)] + ([(rh, rd)] if rd is not None else [])
    outs = [(od, _rows_view(oh, M))] + ([(rd, rh)] if rd is not None else [])
    if want_codes:
        outs += [(cd, ch), (sd, sh)]
    computed = gm in (GAMAX_TENSOR, GAMAX_ROW)
    gh = None
    if computed:
        gh = _gamax_host(gm, gamax, g.numel())
        outs.append((g, gh))

    def launch(r0, r1, st):
        gp = g if (g is None or gm != GAMAX_ROW_GIVEN) else g[r0:]
        return lib.nvfp4_qdq(_ptr(xd[r0]), r1 - r0, K, _x_dtype(x), blk, rnd,
                             _ptr(None if rd is None else rd[r0]), seed, step, row_offset + r0, gm, _ptr(gp),
                             em, bound, _ptr(None if cd is None else cd[r0]), _ptr(None if sd is None else sd[r0]),
                             _ptr(od[r0]), ctypes.c_void_p(st.cuda_stream))

    _pipelined(dev, M, ins, outs, launch, lib, blocking, whole, keep=(g,))
    res = {"out": oh}
    if want_codes:
        res["codes"], res["scales"] = ch, sh
    if computed:
        res["gamax"] = gamax if torch.is_tensor(gamax) and not gamax.is_cuda else gh
    elif g is not None:
        res["gamax"] = g.cpu()
    return res


def _dequantize_pipelined(lib, codes, scales, dev, M, K, gm, g, bound, od_enum, out, blocking=True,
                          whole=False):
    """The host path of nvfp4_dequantize through _pipelined; None when a
    given tensor is not a contiguous row view."""
    chv, shv = _rows_view(codes, M), _rows_view(scales, M)
    odt = torch.bfloat16 if od_enum == BF16 else torch.float32
    if chv is None or shv is None:
        return None
    if not _host_given(out, "out", odt, M * K):
        return None
    oh = _host_out(out, (M, K), odt)
    cd, sd = _empty((M, K // 2), torch.uint8, dev), _empty((M, K // 16), torch.uint8, dev)
    od = _empty((M, K), odt, dev)

    def launch(r0, r1, st):
        gp = g if (g is None or gm != GAMAX_ROW_GIVEN) else g[r0:]
        return lib.nvfp4_dequantize(_ptr(cd[r0]), _ptr(sd[r0]), r1 - r0, K, gm, _ptr(gp), bound, _ptr(od[r0]),
                                    od_enum, ctypes.c_void_p(st.cuda_stream))

    _pipelined(dev, M, [(chv, cd), (shv, sd)], [(od, _rows_view(oh, M))], launch, lib, blocking, whole,
               keep=(g,))
    return oh


def nvfp4_qdq(x: torch.Tensor, *, block="1x16", rounding="rtn", residual=None, seed: int = 0,
              step: int = 0, row_offset: int = 0, gamax_mode="none", gamax=None, err_mode="none",
              scale_bound=None, want_codes: bool = False, out=None, stream=None,
              non_blocking: bool = False) -> dict:
    """quantize then dequantize to bf16 in one pass; ``out`` is bf16 [M,K].
    ``non_blocking`` as for nvfp4_quantize."""
    lib = load_library()
    host = not x.is_cuda
    dev = _device_of(x, residual)
    M, K = x.shape
    blk, rnd = _enum("block", block), _enum("rounding", rounding)
    gm, em = _enum("gamax_mode", gamax_mode), _enum("err_mode", err_mode)
    bound = _default_bound(em, scale_bound)
    if host:
        _host_residual(residual, M, K, dev)
        _non_blocking_stream(non_blocking, stream)
        rows = M >= _PIPE_MIN_ROWS and gm in (GAMAX_NONE, GAMAX_TENSOR_GIVEN, GAMAX_ROW_GIVEN)
        if stream is None and (rows or non_blocking):
            r = _qdq_pipelined(lib, x, dev, M, K, blk, rnd, residual, seed, step, row_offset, gm, gamax, em,
                               bound, out, want_codes, not non_blocking, not rows)
            if r is not None:
                return r
        _non_blocking_refused(non_blocking)
    xd = _host_in(x, dev) if host else x.contiguous()
    rd = _host_in(residual, dev) if host else _dev_residual(residual, dev, M, K)
    g = _gamax_buffer(gm, gamax, M, dev, host)
    o = _out_buf((M, K), torch.bfloat16, out, dev, host, "out")
    codes = _out_buf((M, K // 2), torch.uint8, None, dev, host) if want_codes else None
    scales = _out_buf((M, K // 16), torch.uint8, None, dev, host) if want_codes else None
    if host:
        _inputs_ready(stream)
    with torch.cuda.device(dev):
        rc = lib.nvfp4_qdq(_ptr(xd), M, K, _x_dtype(x), blk, rnd, _ptr(rd), seed, step, row_offset,
                           gm, _ptr(g), em, bound, _ptr(codes), _ptr(scales), _ptr(o),
                           _stream(stream))
    _check(lib, rc)
    res = {"out": o}
    if want_codes:
        res["codes"], res["scales"] = codes, scales
    if g is not None:
        res["gamax"] = g
    if host:
        given = {"out": out}
        if torch.is_tensor(gamax) and not gamax.is_cuda and gm in (GAMAX_TENSOR, GAMAX_ROW):
            given["gamax"] = gamax
        if residual is not None and rd is not residual:
            given["residual"] = residual
            res["residual"] = rd
        res = _finish_host(res, given, stream)
        res.pop("residual", None)
    return res


def nvfp4_dequantize(codes: torch.Tensor, scales: torch.Tensor, M: int, K: int, *,
                     gamax_mode="none", gamax=None, scale_bound=None, out_dtype="bf16", out=None,
                     stream=None, non_blocking: bool = False) -> torch.Tensor:
    """Codes and scale bytes back to values (see nvfp4.h); ``non_blocking`` as
    for nvfp4_quantize."""
    lib = load_library()
    host = not codes.is_cuda
    dev = _device_of(codes, scales)
    gm = _enum("gamax_mode", gamax_mode)
    od = _enum("dtype", out_dtype)
    bound = 448.0 if scale_bound is None else float(scale_bound)
    for t, name, n in ((codes, "codes", M * K // 2), (scales, "scales", M * K // 16)):
        if t.dtype != torch.uint8 or t.numel() != n:
            raise ValueError(f"nvfp4: {name} must be uint8 with {n} elements")
    if not host and scales.device != dev:
        raise ValueError(f"nvfp4: the scales of a call on device codes must be on {dev} (got {scales.device})")
    g = None
    if gm != GAMAX_NONE:
        if gamax is None:
            raise ValueError("gamax_mode needs gamax")
        g = _stage(gamax if torch.is_tensor(gamax) else torch.tensor([float(gamax)]), dev)
        g = g.to(torch.float32).reshape(-1).contiguous()
        need = M if gm in (GAMAX_ROW, GAMAX_ROW_GIVEN) else 1
        if g.numel() < need:
            raise ValueError(f"nvfp4: gamax must hold at least {need} values")
    if host:
        _non_blocking_stream(non_blocking, stream)
    if host and not scales.is_cuda and stream is None and (M >= _PIPE_MIN_ROWS or non_blocking):
        r = _dequantize_pipelined(lib, codes, scales, dev, M, K, gm, g, bound, od, out, not non_blocking,
                                  M < _PIPE_MIN_ROWS)
        if r is not None:
            return r
    if host:
        _non_blocking_refused(non_blocking)
    c = _host_in(codes, dev, "codes") if host else codes.contiguous()
    s = _host_in(scales, dev, "scales") if host else scales.contiguous()
    o = _out_buf((M, K), torch.bfloat16 if od == BF16 else torch.float32, out, dev, host, "out")
    if host:
        _inputs_ready(stream)
    with torch.cuda.device(dev):
        rc = lib.nvfp4_dequantize(_ptr(c), _ptr(s), M, K, gm, _ptr(g), bound, _ptr(o), od,
                                  _stream(stream))
    _check(lib, rc)
    return _finish_host({"o": o}, {"o": out}, stream)["o"] if host else o


def nvfp4_amax(x: torch.Tensor, *, residual=None, per_row: bool = False, out=None,
               stream=None) -> torch.Tensor:
    lib = load_library()
    host = not x.is_cuda
    dev = _device_of(x, residual)
    M, K = x.shape
    if host:
        _host_residual(residual, M, K, dev)
    xd = _host_in(x, dev) if host else x.contiguous()
    rd = _host_in(residual, dev) if host else _dev_residual(residual, dev, M, K)
    need = max(M, 1) if per_row else 1
    # the amax is reduced with device atomics: always a device buffer
    if out is not None and out.is_cuda:
        o = _check_dev(out, "out", torch.float32, need, dev, at_least=True)
    else:
        if out is not None and (out.dtype != torch.float32 or out.numel() < need):
            raise ValueError(f"nvfp4: out must be float32 with at least {need} elements")
        o = _empty((need,), torch.float32, dev)
    if host:
        _inputs_ready(stream)
    with torch.cuda.device(dev):
        rc = lib.nvfp4_amax(_ptr(xd), M, K, _x_dtype(x), _ptr(rd), GAMAX_ROW if per_row else GAMAX_TENSOR,
                            _ptr(o), _stream(stream))
    _check(lib, rc)
    if host or (out is not None and not out.is_cuda):
        return _finish_host({"o": o}, {"o": out}, stream)["o"]
    return o


def nvfp4_scales_to_mma(scales: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """Row-major scale bytes [rows, cols] -> the block-scaled matrix-multiply
    layout, [128*ceil(rows/128), 4*ceil(cols/4)] bytes (see nvfp4.h)."""
    lib = load_library()
    if scales.dim() != 2 or scales.dtype != torch.uint8:
        raise ValueError("nvfp4_scales_to_mma: scales must be a uint8 [rows, cols] tensor")
    host = not scales.is_cuda
    rows, cols = scales.shape
    R, C = -(-rows // 128) * 128, -(-cols // 4) * 4
    if out is not None and not out.is_cuda and not host:
        raise ValueError("nvfp4_scales_to_mma: the output of a call on device scales must be a device tensor")
    if out is not None and not out.is_cuda and (out.dtype != torch.uint8 or out.numel() != R * C):
        raise ValueError(f"nvfp4_scales_to_mma: out must be uint8 with {R * C} elements")
    dev = scales.device if scales.is_cuda else torch.device("cuda", torch.cuda.current_device())
    o = _check_dev(out, "out", torch.uint8, R * C, dev) if out is not None and out.is_cuda else \
        _empty((R, C), torch.uint8, dev)
    s = _stage(scales.contiguous(), dev)
    with torch.cuda.device(dev):
        _check(lib, lib.nvfp4_scales_to_mma(_ptr(s), rows, cols, _ptr(o), _stream(stream)))
    if host or (out is not None and not out.is_cuda):
        return _finish_host({"o": o}, {"o": out}, stream)["o"]
    return o


def nvfp4_mm(codes_a, scales_a, codes_b, scales_b, M: int, N: int, K: int, *, gamax_a=None, gamax_b=None,
             scale_bound: float = 448.0, out_dtype="bf16", out=None, stream=None) -> torch.Tensor:
    """(A B^T) * S_dec(A) * S_dec(B) on the block-scaled FP4 tensor cores;
    scales in the nvfp4_scales_to_mma layout (see nvfp4.h).  Device tensors."""
    lib = load_library()
    odt = _enum("dtype", out_dtype)
    dev = _check_mm_args(codes_a, scales_a, codes_b, scales_b, M, N, K, gamax_a, gamax_b, out, odt)
    o = out if out is not None else _empty((M, N), torch.float32 if odt == F32 else torch.bfloat16, dev)
    with torch.cuda.device(dev):
        rc = lib.nvfp4_mm(_ptr(codes_a), _ptr(scales_a), _ptr(codes_b), _ptr(scales_b), M, N, K, _ptr(gamax_a),
                          _ptr(gamax_b), scale_bound, _ptr(o), odt, _stream(stream))
    _check(lib, rc)
    return o


def _check_mm_args(codes_a, scales_a, codes_b, scales_b, M, N, K, gamax_a, gamax_b, out, odt):
    """nvfp4_mm's tensors, checked before their pointers reach the kernel:
    all on codes_a's CUDA device, contiguous, of their dtype, and (for shapes
    the library accepts: M, N multiples of 128, K of 64) holding at least
    the bytes the product reads or writes.  Shapes the library refuses are
    left to its own EINVAL.  Returns the device."""
    if not torch.is_tensor(codes_a) or not codes_a.is_cuda:
        raise ValueError("nvfp4_mm: the operands must be CUDA tensors")
    dev = codes_a.device
    ok = min(M, N, K) >= 0 and M % 128 == 0 and N % 128 == 0 and K % 64 == 0
    for t, name, n in ((codes_a, "codes_a", M * K // 2), (scales_a, "scales_a", M * K // 16),
                       (codes_b, "codes_b", N * K // 2), (scales_b, "scales_b", N * K // 16)):
        _check_dev(t, name, torch.uint8, n if ok else 0, dev, at_least=True)
    for g, name in ((gamax_a, "gamax_a"), (gamax_b, "gamax_b")):
        if g is not None:
            _check_dev(g, name, torch.float32, 1, dev, at_least=True)
    if out is not None:
        _check_dev(out, "out", torch.float32 if odt == F32 else torch.bfloat16, M * N if ok else 0, dev,
                   at_least=True)
    return dev


def nvfp4_global_scales(gamax: torch.Tensor, scale_bound: float = 448.0, stream=None):
    """(S_enc, S_dec) of each global amax in ``gamax`` (device float32), as
    every quantize / dequantize call computes them (see nvfp4.h)."""
    lib = load_library()
    g = gamax.reshape(-1)
    if not (g.is_cuda and g.dtype == torch.float32 and g.is_contiguous()):
        raise ValueError("nvfp4_global_scales: gamax must be a contiguous CUDA float32 tensor")
    enc, dec = torch.empty_like(g), torch.empty_like(g)
    with torch.cuda.device(g.device):
        _check(lib, lib.nvfp4_global_scales(_ptr(g), g.numel(), float(scale_bound), _ptr(enc), _ptr(dec),
                                            _stream(stream)))
    return enc, dec


def nvfp4_probe_divide(a: torch.Tensor, b: torch.Tensor, stream=None) -> torch.Tensor:
    """Diagnostic: the plain path's device division a / b, elementwise (fp32)."""
    lib = load_library()
    _check_probe_inputs((a, torch.float32, "a"), (b, torch.float32, "b"))
    if a.numel() != b.numel():
        raise ValueError("nvfp4_probe_divide: a and b must hold the same number of values")
    a = a.contiguous()
    b = b.contiguous()
    out = torch.empty_like(a)
    with torch.cuda.device(a.device):
        _check(lib, lib.nvfp4_probe_divide(_ptr(a), _ptr(b), _ptr(out), a.numel(), _stream(stream)))
    return out


def _check_probe_inputs(*specs):
    """A diagnostic's inputs: (tensor, dtype, name) each a CUDA tensor of that
    dtype, all on one device (their pointers go to the kernel as they are)."""
    dev = None
    for t, dtype, name in specs:
        if not torch.is_tensor(t) or not t.is_cuda or t.dtype != dtype:
            raise ValueError(f"nvfp4 probe: {name} must be a CUDA {dtype} tensor")
        if dev is not None and t.device != dev:
            raise ValueError(f"nvfp4 probe: {name} must be on {dev} (got {t.device})")
        dev = t.device


def nvfp4_probe_sub_f16(q: torch.Tensor, v: torch.Tensor, stream=None) -> torch.Tensor:
    """Diagnostic: f16 halves of the int32 words q minus the float32 pairs v,
    rounded once (float32 [2 * q.numel()])."""
    lib = load_library()
    _check_probe_inputs((q, torch.int32, "q"), (v, torch.float32, "v"))
    if v.numel() != 2 * q.numel():
        raise ValueError("nvfp4: q must be int32 words and v float32 with two values per word")
    q = q.contiguous()
    v = v.contiguous()
    out = torch.empty_like(v)
    with torch.cuda.device(v.device):
        _check(lib, lib.nvfp4_probe_sub_f16(_ptr(q), _ptr(v), _ptr(out), q.numel(), _stream(stream)))
    return out


def nvfp4_probe_e2m1(first: int, n: int, out=None, stream=None) -> torch.Tensor:
    """Diagnostic: the device e2m1 codes of the n fp32 bit patterns from
    ``first`` on, packed two per byte (uint8 [(n + 1) // 2])."""
    lib = load_library()
    need = (max(n, 0) + 1) // 2
    if out is not None:
        _check_probe_inputs((out, torch.uint8, "out"))
        o = _check_dev(out, "out", torch.uint8, need, out.device, at_least=True)
    else:
        o = _empty((need,), torch.uint8, torch.device("cuda", torch.cuda.current_device()))
    with torch.cuda.device(o.device):
        _check(lib, lib.nvfp4_probe_e2m1(first, n, _ptr(o), _stream(stream)))
    return o


def nvfp4_last_error() -> str:
    return load_library().nvfp4_last_error().decode()
