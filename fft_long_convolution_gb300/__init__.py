"""Python binding of the fftconv C ABI (include/fftconv.h).

Argument marshalling only: every step of the convolution runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If the
library cannot be loaded, every call raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB_PATH, build as build_library

F16, BF16 = 0, 1
PATH_FUSED, PATH_MULTIPASS = 0, 1
STATUS = {0: "OK", 1: "ERR_INVALID", 2: "ERR_UNSUPPORTED", 3: "ERR_ALIGN", 4: "ERR_WORKSPACE",
          5: "ERR_CUDA", 6: "ERR_ALLOC", 7: "ERR_TIMEOUT"}

EXPORTED = ["fftconv_plan_query", "fftconv_plan_create", "fftconv_plan_destroy", "fftconv_plan_get_info",
            "fftconv_kf_bytes", "fftconv_workspace_bytes", "fftconv_set_workspace", "fftconv_kernel_fft",
            "fftconv_forward", "fftconv_forward_gated", "fftconv_forward_noalloc", "fftconv_host_scratch_bytes",
            "fftconv_forward_host", "fftconv_kernel_fft_adjoint", "fftconv_backward_du",
            "fftconv_backward_du_gated", "fftconv_backward_dk_scratch_bytes", "fftconv_backward_dk",
            "fftconv_partial_scratch_bytes", "fftconv_forward_partial", "fftconv_circular_scratch_bytes",
            "fftconv_forward_circular", "fftconv_selftest_wait", "fftconv_plan_create_sparse",
            "fftconv_plan_get_band", "fftconv_sparse_query", "fftconv_circular_query",
            "fftconv_plan_create_circular",
            "fftconv_device_status", "fftconv_status_string", "fftconv_version"]


class FFTConvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("M", ctypes.c_int64), ("order", ctypes.c_int32),
                ("factors", ctypes.c_int32 * 8), ("path", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("kf_bytes_per_channel", ctypes.c_int64), ("workspace_bytes_per_row", ctypes.c_int64)]

    def as_dict(self):
        return {"N": self.N, "M": self.M, "order": self.order,
                "factors": list(self.factors[: self.order]), "path": self.path, "dtype": self.dtype,
                "kf_bytes_per_channel": self.kf_bytes_per_channel,
                "workspace_bytes_per_row": self.workspace_bytes_per_row}


_lib = None


def lib(auto_build: bool = True):
    """Load (building first if needed) the CUDA library."""
    global _lib
    if _lib is None:
        if auto_build:
            build_library()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"fftconv CUDA library not built: {LIB_PATH}")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        L.fftconv_plan_query.argtypes = [i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(PlanInfo)]
        L.fftconv_plan_create.argtypes = [ctypes.POINTER(vp), i64, ctypes.c_int, ctypes.c_int]
        L.fftconv_plan_create_sparse.argtypes = [ctypes.POINTER(vp), i64, ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
        L.fftconv_sparse_query.argtypes = [i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                           ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                           ctypes.POINTER(ctypes.c_int32)]
        L.fftconv_circular_query.argtypes = [i64, ctypes.c_int, ctypes.POINTER(PlanInfo)]
        L.fftconv_plan_create_circular.argtypes = [ctypes.POINTER(vp), i64, ctypes.c_int]
        L.fftconv_plan_get_band.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                            ctypes.POINTER(ctypes.c_int32)]
        L.fftconv_plan_destroy.argtypes = [vp]
        L.fftconv_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.fftconv_kf_bytes.argtypes = [vp, i64]
        L.fftconv_kf_bytes.restype = sz
        L.fftconv_workspace_bytes.argtypes = [vp, i64, i64]
        L.fftconv_workspace_bytes.restype = sz
        L.fftconv_set_workspace.argtypes = [vp, vp, sz]
        L.fftconv_kernel_fft.argtypes = [vp, vp, vp, i64, vp]
        L.fftconv_forward.argtypes = [vp, vp, vp, vp, i64, i64, vp]
        L.fftconv_forward_gated.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, vp]
        L.fftconv_forward_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, vp]
        L.fftconv_host_scratch_bytes.argtypes = [vp, i64, i64, ctypes.c_int]
        L.fftconv_host_scratch_bytes.restype = sz
        L.fftconv_forward_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, vp, sz, vp]
        L.fftconv_kernel_fft_adjoint.argtypes = [vp, vp, vp, i64, vp]
        L.fftconv_backward_du.argtypes = [vp, vp, vp, vp, i64, i64, vp]
        L.fftconv_backward_du_gated.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, vp]
        L.fftconv_backward_dk_scratch_bytes.argtypes = [vp, i64, i64]
        L.fftconv_backward_dk_scratch_bytes.restype = sz
        L.fftconv_backward_dk.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, vp, sz, vp]
        L.fftconv_partial_scratch_bytes.argtypes = [vp, i64, i64, i64, ctypes.c_int]
        L.fftconv_partial_scratch_bytes.restype = sz
        L.fftconv_forward_partial.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, sz, vp]
        L.fftconv_circular_scratch_bytes.argtypes = [vp, i64, i64, ctypes.c_int]
        L.fftconv_circular_scratch_bytes.restype = sz
        L.fftconv_forward_circular.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, vp, sz, vp]
        L.fftconv_selftest_wait.argtypes = [vp, ctypes.c_int, vp]
        L.fftconv_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
        L.fftconv_status_string.argtypes = [ctypes.c_int]
        L.fftconv_status_string.restype = ctypes.c_char_p
        L.fftconv_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(st: int, what: str):
    if st != 0:
        raise FFTConvError(st, what)


def query(N: int, dtype: int, order: int = 0) -> dict:
    info = PlanInfo()
    _check(lib().fftconv_plan_query(N, dtype, order, ctypes.byref(info)), "fftconv_plan_query")
    return info.as_dict()


def circular_query(C: int, dtype: int) -> dict:
    """The plan a circular convolution of length C would use (no GPU)."""
    info = PlanInfo()
    _check(lib().fftconv_circular_query(C, dtype, ctypes.byref(info)), "fftconv_circular_query")
    return info.as_dict()


def sparse_query(N: int, dtype: int, band, order: int = 0) -> dict:
    """Pairs of sub-rows a frequency-sparse plan would transform (no GPU)."""
    arr = (ctypes.c_int32 * max(1, len(band)))(*[int(b) for b in band])
    run, tot = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().fftconv_sparse_query(N, dtype, order, arr, len(band), ctypes.byref(run), ctypes.byref(tot)),
           "fftconv_sparse_query")
    return {"pairs_run": run.value, "pairs_total": tot.value}


def _dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.float16:
        return F16
    if torch_dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {torch_dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Plan:
    """A plan for one sequence length N and dtype (torch.float16 / bfloat16)."""

    def __init__(self, N: int, dtype, order: int = 0, band=None, circular: bool = False):
        """band: one int per factor (outer first) for a frequency-sparse plan;
        None for the dense convolution.  circular: a plan for the circular
        convolution of length N (rows of N samples, k of N taps)."""
        self.N = int(N)
        self.torch_dtype = dtype
        self.dtype = _dtype_code(dtype)
        self.circular = bool(circular)
        h = ctypes.c_void_p()
        if circular:
            if band is not None or order != 0:
                raise ValueError("a circular plan takes no band and no order")
            _check(lib().fftconv_plan_create_circular(ctypes.byref(h), self.N, self.dtype),
                   "fftconv_plan_create_circular")
        elif band is None:
            _check(lib().fftconv_plan_create(ctypes.byref(h), self.N, self.dtype, order), "fftconv_plan_create")
        else:
            arr = (ctypes.c_int32 * max(1, len(band)))(*[int(b) for b in band])
            _check(lib().fftconv_plan_create_sparse(ctypes.byref(h), self.N, self.dtype, order, arr, len(band)),
                   "fftconv_plan_create_sparse")
        self._h = h
        info = PlanInfo()
        _check(lib().fftconv_plan_get_info(self._h, ctypes.byref(info)), "fftconv_plan_get_info")
        self.info = info.as_dict()
        self._workspace = None
        self._host_scratch = None

    def band(self) -> dict:
        """The plan's band per factor and the pass-B pairs that run / exist."""
        b = (ctypes.c_int32 * 8)()
        run, tot = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().fftconv_plan_get_band(self._h, b, ctypes.byref(run), ctypes.byref(tot)), "fftconv_plan_get_band")
        return {"band": list(b[: self.info["order"]]), "pairs_run": run.value, "pairs_total": tot.value}

    def close(self):
        if getattr(self, "_h", None):
            lib().fftconv_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def kf_bytes(self, H: int) -> int:
        return int(lib().fftconv_kf_bytes(self._h, H))

    def workspace_bytes(self, B: int, H: int) -> int:
        return int(lib().fftconv_workspace_bytes(self._h, B, H))

    def set_workspace(self, buf) -> None:
        """Attach a caller-owned device buffer (a torch tensor kept alive here)."""
        self._workspace = buf
        n = 0 if buf is None else buf.numel() * buf.element_size()
        _check(lib().fftconv_set_workspace(self._h, _ptr(buf), n), "fftconv_set_workspace")

    def kernel_fft(self, k, k_f=None, stream=None):
        """k: float32 [H, N] on the GPU -> opaque k_f (uint8 tensor)."""
        import torch
        H = k.shape[0]
        if k.dtype != torch.float32 or not k.is_contiguous() or k.shape[-1] != self.N:
            raise ValueError("k must be contiguous float32 [H, N]")
        if k_f is None:
            k_f = torch.empty(self.kf_bytes(H), dtype=torch.uint8, device=k.device)
        _check(lib().fftconv_kernel_fft(self._h, _ptr(k), _ptr(k_f), H, _stream(stream)), "fftconv_kernel_fft")
        return k_f

    def _ensure_workspace(self, B, H, device):
        import torch
        need = self.workspace_bytes(B, H)
        if need and (self._workspace is None or self._workspace.numel() < need):
            self.set_workspace(torch.empty(need, dtype=torch.uint8, device=device))

    def forward(self, u, k_f, y=None, stream=None):
        """u: [B, H, N] (plan dtype, GPU) -> y = causal conv with k."""
        import torch
        B, H, N = u.shape
        if y is None:
            y = torch.empty_like(u)
        self._ensure_workspace(B, H, u.device)
        _check(lib().fftconv_forward(self._h, _ptr(u), _ptr(k_f), _ptr(y), B, H, _stream(stream)),
               "fftconv_forward")
        return y

    def forward_gated(self, u, w_in, w_out, k_f, y=None, stream=None):
        """y = w_out * conv(u * w_in, k)."""
        import torch
        B, H, N = u.shape
        if y is None:
            y = torch.empty_like(u)
        self._ensure_workspace(B, H, u.device)
        _check(lib().fftconv_forward_gated(self._h, _ptr(u), _ptr(w_in), _ptr(w_out), _ptr(k_f), _ptr(y),
                                           B, H, _stream(stream)), "fftconv_forward_gated")
        return y

    def forward_host(self, u, k_f, w_in=None, w_out=None, y=None, stream=None):
        """u (and w_in, w_out): host tensors [B, H, N] in the plan dtype,
        page-locked for the copies to overlap -> y (host).  Chunks of rows are
        copied in, convolved and copied back with the three steps overlapped;
        y is complete once the stream has been synchronised."""
        import torch
        for t in (u, w_in, w_out, y):
            if t is not None and (t.is_cuda or not t.is_contiguous() or t.dtype != self.torch_dtype):
                raise ValueError("host tensors must be contiguous CPU tensors of the plan dtype")
        if (w_in is None) != (w_out is None):
            raise ValueError("w_in and w_out go together")
        B, H, N = u.shape
        if y is None:
            y = torch.empty(u.shape, dtype=u.dtype, pin_memory=True)
        gated = w_in is not None
        need = int(lib().fftconv_host_scratch_bytes(self._h, B, H, int(gated)))
        if need and (self._host_scratch is None or self._host_scratch.numel() < need):
            self._host_scratch = torch.empty(need, dtype=torch.uint8, device=k_f.device)
        n = 0 if self._host_scratch is None else self._host_scratch.numel()
        _check(lib().fftconv_forward_host(self._h, _ptr(u), _ptr(w_in), _ptr(w_out), _ptr(k_f), _ptr(y), B, H,
                                          _ptr(self._host_scratch), n, _stream(stream)), "fftconv_forward_host")
        return y

    # ---- partial convolution (kernels of at most N/2 taps, sequences of any multiple of N/2)

    def kernel_fft_partial(self, k, k_f=None, stream=None):
        """k: float32 [H, T] with T <= N/2 taps -> k_f for forward_partial."""
        import torch
        H, T = k.shape
        if T > self.N // 2:
            raise ValueError(f"a partial-convolution kernel has at most {self.N // 2} taps")
        kp = torch.zeros(H, self.N, dtype=torch.float32, device=k.device)
        kp[:, :T] = k
        return self.kernel_fft(kp, k_f=k_f, stream=stream)

    def forward_partial(self, u, k_f, w_in=None, w_out=None, y=None, stream=None):
        """u: [B, H, N'] with N' a multiple of N/2 -> the causal convolution with
        the kernel of kernel_fft_partial (gated when w_in, w_out are given)."""
        import torch
        B, H, Np = u.shape
        if y is None:
            y = torch.empty_like(u)
        gated = w_in is not None
        need = int(lib().fftconv_partial_scratch_bytes(self._h, B, H, Np, int(gated)))
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=u.device)
        _check(lib().fftconv_forward_partial(self._h, _ptr(u), _ptr(w_in), _ptr(w_out), _ptr(k_f), _ptr(y), B, H, Np,
                                             _ptr(scratch), need, _stream(stream)), "fftconv_forward_partial")
        return y

    def forward_circular(self, u, k_f, w_in=None, w_out=None, y=None, stream=None):
        """u: [B, H, N/2] -> circular convolution of length N/2 with the kernel
        of kernel_fft_partial (its N/2 taps)."""
        import torch
        B, H, C = u.shape
        if C != self.N // 2:
            raise ValueError(f"circular length must be {self.N // 2} for this plan")
        if y is None:
            y = torch.empty_like(u)
        gated = w_in is not None
        need = int(lib().fftconv_circular_scratch_bytes(self._h, B, H, int(gated)))
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=u.device)
        _check(lib().fftconv_forward_circular(self._h, _ptr(u), _ptr(w_in), _ptr(w_out), _ptr(k_f), _ptr(y), B, H,
                                              _ptr(scratch), need, _stream(stream)), "fftconv_forward_circular")
        return y

    # ---- backward (gradients in u and k)

    def kernel_fft_adjoint(self, k, k_f=None, stream=None):
        """k: float32 [H, N] -> opaque adjoint k_f (correlation with k)."""
        import torch
        H = k.shape[0]
        if k.dtype != torch.float32 or not k.is_contiguous() or k.shape[-1] != self.N:
            raise ValueError("k must be contiguous float32 [H, N]")
        if k_f is None:
            k_f = torch.empty(self.kf_bytes(H), dtype=torch.uint8, device=k.device)
        _check(lib().fftconv_kernel_fft_adjoint(self._h, _ptr(k), _ptr(k_f), H, _stream(stream)),
               "fftconv_kernel_fft_adjoint")
        return k_f

    def backward_du(self, dy, k_f_adj, w_in=None, w_out=None, du=None, stream=None):
        """du = corr(dy, k) (gated: w_in * corr(w_out * dy, k))."""
        import torch
        B, H, N = dy.shape
        if du is None:
            du = torch.empty_like(dy)
        self._ensure_workspace(B, H, dy.device)
        if w_in is None:
            st = lib().fftconv_backward_du(self._h, _ptr(dy), _ptr(k_f_adj), _ptr(du), B, H, _stream(stream))
        else:
            st = lib().fftconv_backward_du_gated(self._h, _ptr(dy), _ptr(w_in), _ptr(w_out), _ptr(k_f_adj),
                                                 _ptr(du), B, H, _stream(stream))
        _check(st, "fftconv_backward_du")
        return du

    def backward_dk(self, u, dy, w_in=None, w_out=None, dk=None, stream=None):
        """dk [H, N] float32 = sum_b corr(w_out * dy_b, w_in * u_b)."""
        import torch
        B, H, N = u.shape
        if dk is None:
            dk = torch.empty(H, N, dtype=torch.float32, device=u.device)
        need = int(lib().fftconv_backward_dk_scratch_bytes(self._h, B, H))
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=u.device)
        _check(lib().fftconv_backward_dk(self._h, _ptr(u), _ptr(dy), _ptr(w_in), _ptr(w_out), _ptr(dk), B, H,
                                         _ptr(scratch), need, _stream(stream)), "fftconv_backward_dk")
        return dk

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int()
        _check(lib().fftconv_device_status(self._h, _stream(stream), ctypes.byref(v)), "fftconv_device_status")
        return v.value


def status_string(code: int) -> str:
    return lib().fftconv_status_string(code).decode()
