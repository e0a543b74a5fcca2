"""SNACK truly-sparse linear layer on GB300: Python binding of libsnack.so.

Argument marshalling only.  Every operation runs in the library's CUDA
kernels; PyTorch provides device memory and streams.  The function names are
those of the C ABI (include/snack.h):

    h = snack_create(out, in, row, col, val)          # COO in any order
    Y = snack_forward(h, X)                           # Y  = X W^T
    dX = snack_backward_input(h, dY)                  # dX = dY W
    dW = snack_backward_weight(h, X, dY)              # dW[k] at stored k
    dX, dW = snack_backward(h, X, dY)                 # both, one dY transpose
    snack_prune_regrow(h, frac, seed)                 # Appendix G topology step
    snack_values(h)                                   # torch view of the values

Tensors are fp32, contiguous, on the handle's device; results are written to
the given output tensors (or new ones) on the current torch CUDA stream unless
`stream` is given.  A C-ABI error raises SnackError.  ``SnackLinear`` is a thin
nn.Module / autograd wrapper for training loops.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _abi

_lib = _abi.load()

__all__ = [
    "SnackError", "SnackHandle", "snack_create", "snack_create_random", "snack_forward",
    "snack_backward_input", "snack_backward_weight", "snack_backward", "snack_prune_regrow",
    "snack_values", "snack_values_changed", "snack_sgd_step", "snack_adam_step", "snack_optimizer_state", "snack_export", "snack_export_segments", "snack_plan", "snack_nnz",
    "snack_device_bytes", "snack_destroy", "snack_launch_count", "snack_debug_fail_alloc", "snack_forward_csr_static", "snack_device_error", "snack_selftest_wait", "SnackLinear", "library_path",
]


def library_path() -> str:
    return _abi.LIB_PATH


class SnackError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_abi.STATUS.get(status, status)}: {message}")
        self.status = status


class SnackHandle:
    """Owns one C handle; destroyed when garbage-collected."""

    def __init__(self, ptr: int, out: int, inp: int, device: torch.device):
        self.ptr = ctypes.c_void_p(ptr)
        self.out = out
        self.inp = inp
        self.device = device

    @property
    def nnz(self) -> int:
        return int(_lib.snack_nnz(self.ptr))

    def close(self):
        if self.ptr is not None and self.ptr.value:
            _lib.snack_destroy(self.ptr)
        self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check(status: int, h: SnackHandle | None = None):
    if status != 0:
        msg = _lib.snack_last_error(h.ptr if h is not None else None)
        raise SnackError(status, (msg or b"").decode(errors="replace"))


def _stream(stream, device=None):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev_f32(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host_or_dev(a, dtype):
    """(pointer, on_device, keepalive) for an index / value array."""
    if isinstance(a, torch.Tensor):
        want = torch.int32 if dtype == np.int32 else torch.float32
        t = a.to(want).contiguous() if a.dtype != want or not a.is_contiguous() else a
        return ctypes.c_void_p(t.data_ptr()), bool(t.is_cuda), t
    arr = np.ascontiguousarray(a, dtype=dtype)
    return ctypes.c_void_p(arr.ctypes.data), False, arr


def snack_create(out: int, inp: int, row, col, val=None, stream=None) -> SnackHandle:
    """Build a layer from a COO triple in any order (host numpy or CUDA tensors)."""
    rp, rdev, rk = _host_or_dev(row, np.int32)
    cp, cdev, ck = _host_or_dev(col, np.int32)
    nnz = int(rk.numel() if isinstance(rk, torch.Tensor) else rk.size)
    vp, vdev, vk = (None, rdev, None) if val is None else _host_or_dev(val, np.float32)
    if not (rdev == cdev == vdev):
        raise ValueError("row, col and val must all be host arrays or all CUDA tensors")
    dev = torch.device("cuda", torch.cuda.current_device())
    h = ctypes.c_void_p()
    _check(_lib.snack_create(out, inp, nnz, rp if nnz else None, cp if nnz else None,
                             vp if nnz else None, int(rdev), _stream(stream), ctypes.byref(h)))
    return SnackHandle(h.value, out, inp, dev)


def snack_create_random(out: int, inp: int, nnz: int, seed: int, stream=None):
    """Layer with nnz cells drawn by Algorithm 2 on the device (values 0).

    Returns (handle, trials)."""
    h = ctypes.c_void_p()
    trials = ctypes.c_int64(0)
    _check(_lib.snack_create_random(out, inp, nnz, seed & (2**64 - 1), _stream(stream),
                                    ctypes.byref(h), ctypes.byref(trials)))
    dev = torch.device("cuda", torch.cuda.current_device())
    return SnackHandle(h.value, out, inp, dev), int(trials.value)


def _batch(t: torch.Tensor, width: int, name: str) -> int:
    if t.dim() != 2 or t.shape[1] != width:
        raise ValueError(f"{name} must be [batch][{width}], got {tuple(t.shape)}")
    return int(t.shape[0])


def snack_forward(h: SnackHandle, X: torch.Tensor, Y: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Y = X W^T."""
    X = _dev_f32(X, "X")
    B = _batch(X, h.inp, "X")
    if Y is None:
        Y = torch.empty((B, h.out), dtype=torch.float32, device=X.device)
    _dev_f32(Y, "Y")
    _check(_lib.snack_forward(h.ptr, _ptr(X), _ptr(Y), B, _stream(stream, X.device)), h)
    return Y


def snack_backward_input(h: SnackHandle, dY: torch.Tensor, dX: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """dX = dY W."""
    dY = _dev_f32(dY, "dY")
    B = _batch(dY, h.out, "dY")
    if dX is None:
        dX = torch.empty((B, h.inp), dtype=torch.float32, device=dY.device)
    _dev_f32(dX, "dX")
    _check(_lib.snack_backward_input(h.ptr, _ptr(dY), _ptr(dX), B, _stream(stream, dY.device)), h)
    return dX


def snack_backward_weight(h: SnackHandle, X: torch.Tensor, dY: torch.Tensor,
                          dW: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dW[k] = sum_b dY[b,row_k] X[b,col_k] (canonical order)."""
    X, dY = _dev_f32(X, "X"), _dev_f32(dY, "dY")
    B = _batch(X, h.inp, "X")
    if _batch(dY, h.out, "dY") != B:
        raise ValueError("X and dY batch sizes differ")
    if dW is None:
        dW = torch.empty(h.nnz, dtype=torch.float32, device=X.device)
    _dev_f32(dW, "dW")
    _check(_lib.snack_backward_weight(h.ptr, _ptr(X), _ptr(dY), _ptr(dW), B,
                                      _stream(stream, X.device)), h)
    return dW


def snack_backward(h: SnackHandle, X: torch.Tensor | None, dY: torch.Tensor,
                   dX: torch.Tensor | None = None, dW: torch.Tensor | None = None,
                   need_dx: bool = True, need_dw: bool = True, stream=None):
    """(dX, dW) sharing one transposed dY; either may be skipped."""
    dY = _dev_f32(dY, "dY")
    B = _batch(dY, h.out, "dY")
    if need_dx and dX is None:
        dX = torch.empty((B, h.inp), dtype=torch.float32, device=dY.device)
    if need_dw and dW is None:
        dW = torch.empty(h.nnz, dtype=torch.float32, device=dY.device)
    if need_dw:
        X = _dev_f32(X, "X")
        if _batch(X, h.inp, "X") != B:
            raise ValueError("X and dY batch sizes differ")
    _check(_lib.snack_backward(h.ptr, _ptr(X) if need_dw else None, _ptr(dY),
                               _ptr(dX) if need_dx else None, _ptr(dW) if need_dw else None, B,
                               _stream(stream, dY.device)), h)
    return (dX if need_dx else None), (dW if need_dw else None)


def snack_prune_regrow(h: SnackHandle, frac: float, seed: int, stream=None):
    """Magnitude prune + uniform regrow.  Returns (pruned, trials)."""
    p = ctypes.c_int64(0)
    t = ctypes.c_int64(0)
    _check(_lib.snack_prune_regrow(h.ptr, ctypes.c_float(frac), seed & (2**64 - 1),
                                   _stream(stream), ctypes.byref(p), ctypes.byref(t)), h)
    return int(p.value), int(t.value)


class _CudaArray:
    def __init__(self, ptr: int, n: int, keep):
        self._keep = keep
        self.__cuda_array_interface__ = {
            "shape": (n,), "typestr": "<f4", "data": (ptr, False), "version": 3, "strides": None}


def snack_values(h: SnackHandle) -> torch.Tensor:
    """The stored values (canonical order) as a CUDA tensor sharing the handle's memory."""
    p = ctypes.c_void_p()
    _check(_lib.snack_values(h.ptr, ctypes.byref(p)), h)
    n = h.nnz
    if n == 0:
        return torch.empty(0, dtype=torch.float32, device=h.device)
    return torch.as_tensor(_CudaArray(p.value, n, h), device=h.device)


def snack_values_changed(h: SnackHandle, stream=None) -> None:
    """Declare that writes through the snack_values() view are done: the
    handle re-derives its column-ordered value copy and dX streams it again."""
    _check(_lib.snack_values_changed(h.ptr, _stream(stream, h.device)), h)


def _opt_inputs(h: SnackHandle, X: torch.Tensor, dY: torch.Tensor):
    X, dY = _dev_f32(X, "X"), _dev_f32(dY, "dY")
    B = _batch(X, h.inp, "X")
    if _batch(dY, h.out, "dY") != B:
        raise ValueError("X and dY batch sizes differ")
    return X, dY, B


def snack_sgd_step(h: SnackHandle, X: torch.Tensor, dY: torch.Tensor, lr: float,
                   momentum: float = 0.0, weight_decay: float = 0.0, stream=None) -> None:
    """One SGD step on the stored values from their gradient
    sum_b dY[b,row_k] X[b,col_k] (never returned; batches of 1-4 compute it
    inside the step's kernel, larger ones in the handle's gradient buffer)."""
    X, dY, B = _opt_inputs(h, X, dY)
    _check(_lib.snack_sgd_step(h.ptr, _ptr(X), _ptr(dY), B, lr, momentum, weight_decay,
                               _stream(stream, X.device)), h)


def snack_adam_step(h: SnackHandle, X: torch.Tensor, dY: torch.Tensor, lr: float = 1e-3,
                    betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0,
                    step: int = 1, stream=None) -> None:
    """One Adam step (step = t >= 1) on the stored values from their
    gradient (as for snack_sgd_step)."""
    X, dY, B = _opt_inputs(h, X, dY)
    _check(_lib.snack_adam_step(h.ptr, _ptr(X), _ptr(dY), B, lr, betas[0], betas[1], eps,
                                weight_decay, step, _stream(stream, X.device)), h)


def snack_optimizer_state(h: SnackHandle, which: int) -> torch.Tensor:
    """Optimizer state array `which` (0: momentum / first moment, 1: second
    moment) as a CUDA tensor sharing the handle's memory (canonical order)."""
    p = ctypes.c_void_p()
    _check(_lib.snack_optimizer_state(h.ptr, which, ctypes.byref(p)), h)
    return torch.as_tensor(_CudaArray(p.value, h.nnz, h), device=h.device)


def snack_export(h: SnackHandle):
    """(row, col, val) numpy arrays in canonical order."""
    n = h.nnz
    row = np.empty(n, np.int32)
    col = np.empty(n, np.int32)
    val = np.empty(n, np.float32)
    _check(_lib.snack_export(h.ptr, ctypes.c_void_p(row.ctypes.data),
                             ctypes.c_void_p(col.ctypes.data), ctypes.c_void_p(val.ctypes.data),
                             0, _stream(None)), h)
    return row, col, val


def snack_export_segments(h: SnackHandle):
    """dict(row_ptr, col_ptr, csc_row, csc_perm) as numpy arrays."""
    n = h.nnz
    res = dict(row_ptr=np.empty(h.out + 1, np.int32), col_ptr=np.empty(h.inp + 1, np.int32),
               csc_row=np.empty(n, np.int32), csc_perm=np.empty(n, np.int32))
    _check(_lib.snack_export_segments(h.ptr, *[ctypes.c_void_p(res[k].ctypes.data) for k in
                                               ("row_ptr", "col_ptr", "csc_row", "csc_perm")],
                                      _stream(None)), h)
    return res


def snack_plan(h: SnackHandle, op: int, batch: int, with_resident: bool = False):
    """(slice_width, lanes_per_segment, segments[, resident]) chosen for op
    0/1/2 at this batch; resident = 1 when every block holds the whole dense
    operand in shared memory."""
    w, l, s, t = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
    _check(_lib.snack_plan(h.ptr, op, batch, ctypes.byref(w), ctypes.byref(l), ctypes.byref(s),
                           ctypes.byref(t)), h)
    if with_resident:
        return int(w.value), int(l.value), int(s.value), int(t.value)
    return int(w.value), int(l.value), int(s.value)


def snack_forward_csr_static(out: int, inp: int, row_ptr: torch.Tensor, col: torch.Tensor,
                             val: torch.Tensor, X: torch.Tensor, Y: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """Y = X W^T from caller-held CSR arrays, with the library's fixed device
    scratch instead of any allocation (for callers that cannot allocate when
    they run the layer).  Allocates Y only if it is not given."""
    X = _dev_f32(X, "X")
    B = _batch(X, inp, "X")
    for t, name, dt in ((row_ptr, "row_ptr", torch.int32), (col, "col", torch.int32),
                        (val, "val", torch.float32)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dt and t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous CUDA {dt} tensor")
    if Y is None:
        Y = torch.empty((B, out), dtype=torch.float32, device=X.device)
    _dev_f32(Y, "Y")
    nnz = int(col.numel())
    _check(_lib.snack_forward_csr_static(out, inp, nnz, _ptr(row_ptr), _ptr(col) if nnz else None,
                                         _ptr(val) if nnz else None, _ptr(X), _ptr(Y), B,
                                         _stream(stream, X.device)))
    return Y


def snack_selftest_wait(stream=None) -> int:
    """Run the bounded-wait self-test (a wait nothing completes); returns 1
    when the wait gave up as designed."""
    flag = ctypes.c_int(0)
    _check(_lib.snack_selftest_wait(_stream(stream), ctypes.byref(flag)))
    return int(flag.value)


def snack_device_error(h: SnackHandle) -> int:
    """Read and clear the handle's device error flag (1 = a bounded wait gave up)."""
    f = ctypes.c_int(0)
    _check(_lib.snack_device_error(h.ptr, ctypes.byref(f), _stream(None)), h)
    return int(f.value)


def snack_debug_fail_alloc(after: int) -> None:
    """Test hook: after `after` more device allocations by the library, one
    fails as out of memory (the hook then disarms); negative disarms."""
    _lib.snack_debug_fail_alloc(int(after))


def snack_launch_count() -> int:
    """Kernel launches issued by the library in this process so far."""
    return int(_lib.snack_launch_count())


def snack_nnz(h: SnackHandle) -> int:
    return h.nnz


def snack_device_bytes(h: SnackHandle) -> int:
    return int(_lib.snack_device_bytes(h.ptr))


def snack_destroy(h: SnackHandle):
    h.close()


class _SnackFunction(torch.autograd.Function):
    """Forward Y = X W^T; backward dX = dY W and dW at the stored entries.

    The values tensor is saved with X, so autograd refuses a backward after
    the values were changed in place between forward and backward."""

    @staticmethod
    def forward(ctx, X, values, handle):
        ctx.handle = handle
        ctx.save_for_backward(X, values)
        return snack_forward(handle, X.contiguous())

    @staticmethod
    def backward(ctx, dY):
        X, _ = ctx.saved_tensors
        need_dx, need_dw = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (need_dx or need_dw):
            return None, None, None
        dX, dW = snack_backward(ctx.handle, X.contiguous(), dY.contiguous(), need_dx=need_dx,
                                need_dw=need_dw)
        return dX, dW, None


class SnackLinear(torch.nn.Module):
    """Drop-in for nn.Linear whose weight exists only as its stored entries.

    ``weight_values`` is a Parameter viewing the library's value array
    (canonical order: rows ascending, columns ascending within a row), so a
    torch optimizer updates the layer in place and its gradient arrives in
    the same order.  Bias (optional) is a dense Parameter added by PyTorch;
    it is not part of the sparse product.

    The library keeps a column-ordered copy of the values for dX.  While the
    values change every step (training this layer), dX reads them through
    the column permutation instead: re-deriving the copy after each update
    costs more than the permuted reads it saves (10000x10000 at 95 %,
    forward + dX + Adam step: 72 us through the permutation, 83 us with the
    copy re-derived after the step, batch 1).  When the values stay the same
    from one forward to the next (a frozen layer whose input gradient is
    still needed), the module has the copy re-derived once and dX streams
    it; the first write after that (the tensor's version counter moves)
    makes the copy stale again before any dX can read it."""

    def __init__(self, in_features: int, out_features: int, nnz: int, seed: int,
                 std: float = 0.02, bias: bool = True):
        super().__init__()
        self.in_features, self.out_features = in_features, out_features
        self.handle, _ = snack_create_random(out_features, in_features, nnz, seed)
        vals = snack_values(self.handle)
        g = torch.Generator(device="cpu").manual_seed(seed)
        vals.copy_((torch.randn(nnz, generator=g) * std).to(vals.device))
        self.weight_values = torch.nn.Parameter(vals)
        self.bias = torch.nn.Parameter(torch.zeros(out_features, device=vals.device)) if bias else None
        self._seen_version = None   # version of weight_values at the last forward
        self._copy_current = False  # the library's column-ordered copy is trusted

    @property
    def nnz(self) -> int:
        return self.handle.nnz

    def sync_values(self) -> None:
        """Keep the library's column-ordered value copy consistent with
        ``weight_values`` (called by forward): values written since the last
        forward make it stale (dX reads through the permutation); values
        unchanged since the last forward have it re-derived once."""
        v = self.weight_values._version
        if v != self._seen_version:
            if self._copy_current:
                snack_values(self.handle)  # marks the copy stale
                self._copy_current = False
            self._seen_version = v
        elif not self._copy_current:
            snack_values_changed(self.handle)
            self._copy_current = True

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        self.sync_values()
        shape = x.shape
        y = _SnackFunction.apply(x.reshape(-1, self.in_features), self.weight_values, self.handle)
        y = y.reshape(*shape[:-1], self.out_features)
        return y + self.bias if self.bias is not None else y

    @torch.no_grad()
    def prune_regrow(self, frac: float, seed: int):
        """Topology step in place (magnitude prune + Algorithm 2 regrow,
        canonical order restored).  ``weight_values`` keeps its storage and
        now holds the survivors' values and zeros for the regrown entries,
        in the new canonical order.  Optimizer state that torch keeps per
        element of ``weight_values`` (momentum, Adam moments) is NOT
        reordered: reset it after this call, or train with the library's
        own steps (snack_sgd_step / snack_adam_step), whose state follows the
        entries.  Returns (pruned, trials)."""
        return snack_prune_regrow(self.handle, frac, seed)

    def export(self):
        """(row, col, val) numpy arrays of the stored entries in canonical order."""
        return snack_export(self.handle)
