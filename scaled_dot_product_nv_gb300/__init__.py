"""Python binding of the nv_sdpa C ABI (include/nv_sdpa.h): argument marshalling only.

Every step of the attention forward runs in the CUDA kernels of libnvsdpa.so; this
module converts Python arguments to C ones and raises on a non-OK status.  There is
no CPU path: if the library is missing, loading it raises.

Raw entry points (same names as the C functions, pointers as ints):
    nv_sdpa, nv_sdpa_plan, nv_sdpa_host, nv_sdpa_noalloc, nv_sdpa_device_status,
    nv_sdpa_set_wait_limit, nv_sdpa_status_string, nv_sdpa_abi_version
Torch convenience (torch tensors for device memory and the current stream):
    sdpa(q, k, v, mask_kind=..., scale=..., bool_mask=None, sinks=None)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvsdpa.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
MASKS = {"none": 0, "causal": 1, "bool": 2}
PATHS = {0: "noop", 1: "no_keys", 2: "prefill", 3: "decode"}
KERNELS = {0: "none", 1: "fill", 2: "prefill_tc", 3: "tiled_simt", 4: "decode_mma"}


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "Hq", "Hkv", "Lq", "Lk", "d", "dv")]


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("nblk", ctypes.c_int64), ("keys_per_blk", ctypes.c_int64),
                ("rows_per_cta", ctypes.c_int64), ("grid", ctypes.c_int64),
                ("launches", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64)]

    def as_dict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["path"] = PATHS.get(self.path, self.path)
        d["kernel"] = KERNELS.get(self.kernel, self.kernel)
        return d


class NvSdpaError(RuntimeError):
    def __init__(self, status: int, what: str = "nv_sdpa"):
        self.status = status
        super().__init__(f"{what}: status {status} ({nv_sdpa_status_string(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"nv_sdpa CUDA library not built ({LIB_PATH} missing); "
                               "run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, u8p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p
        sig = [vp, vp, vp, ctypes.POINTER(Dims), ctypes.c_int, u8p, vp, ctypes.c_float,
               vp, vp, ctypes.c_int, vp]
        L.nv_sdpa.argtypes = sig
        L.nv_sdpa.restype = ctypes.c_int
        L.nv_sdpa_host.argtypes = sig
        L.nv_sdpa_host.restype = ctypes.c_int
        L.nv_sdpa_noalloc.argtypes = sig
        L.nv_sdpa_noalloc.restype = ctypes.c_int
        L.nv_sdpa_plan.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(Plan)]
        L.nv_sdpa_plan.restype = ctypes.c_int
        L.nv_sdpa_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.nv_sdpa_device_status.restype = ctypes.c_int
        L.nv_sdpa_set_wait_limit.argtypes = [ctypes.c_uint64]
        L.nv_sdpa_set_wait_limit.restype = ctypes.c_int
        L.nv_sdpa_status_string.argtypes = [ctypes.c_int]
        L.nv_sdpa_status_string.restype = ctypes.c_char_p
        L.nv_sdpa_abi_version.argtypes = []
        L.nv_sdpa_abi_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _dims(B, Hq, Hkv, Lq, Lk, d, dv) -> Dims:
    return Dims(B, Hq, Hkv, Lq, Lk, d, dv)


def nv_sdpa(q, k, v, dims, mask_kind, bool_mask, sinks, scale, out, lse, dtype, stream) -> int:
    """The C call; pointers are ints (0 = NULL), dims a Dims or a 7-tuple."""
    if not isinstance(dims, Dims):
        dims = _dims(*dims)
    return lib().nv_sdpa(q, k, v, ctypes.byref(dims), int(mask_kind), bool_mask or None,
                         sinks or None, ctypes.c_float(scale), out, lse or None, int(dtype),
                         stream or None)


def nv_sdpa_host(q, k, v, dims, mask_kind, bool_mask, sinks, scale, out, lse, dtype, stream) -> int:
    if not isinstance(dims, Dims):
        dims = _dims(*dims)
    return lib().nv_sdpa_host(q, k, v, ctypes.byref(dims), int(mask_kind), bool_mask or None,
                              sinks or None, ctypes.c_float(scale), out, lse or None, int(dtype),
                              stream or None)


def nv_sdpa_noalloc(q, k, v, dims, mask_kind, bool_mask, sinks, scale, out, lse, dtype, stream) -> int:
    """nv_sdpa for callers that cannot allocate device memory: scratch comes from the
    library's fixed device array (STATIC_SCRATCH_BYTES); calls that overlap on the GPU
    share it and must be serialised by the caller."""
    if not isinstance(dims, Dims):
        dims = _dims(*dims)
    return lib().nv_sdpa_noalloc(q, k, v, ctypes.byref(dims), int(mask_kind), bool_mask or None,
                                 sinks or None, ctypes.c_float(scale), out, lse or None, int(dtype),
                                 stream or None)


def _header_define(name: str) -> int:
    """An integer #define of the C header (so that the binding never restates a value)."""
    import re
    path = os.path.join(os.path.dirname(_PKG), "include", "nv_sdpa.h")
    with open(path) as f:
        m = re.search(r"#define\s+" + name + r"\s+\((\d+)u?\s*<<\s*(\d+)\)|#define\s+" + name +
                      r"\s+(\d+)", f.read())
    if not m:
        raise RuntimeError(f"{name} not found in {path}")
    return int(m.group(1)) << int(m.group(2)) if m.group(1) else int(m.group(3))


STATIC_SCRATCH_BYTES = _header_define("NV_SDPA_STATIC_SCRATCH_BYTES")


def nv_sdpa_plan(dims, mask_kind, has_sinks, dtype):
    """Returns (status, plan dict or None)."""
    if not isinstance(dims, Dims):
        dims = _dims(*dims)
    pl = Plan()
    st = lib().nv_sdpa_plan(ctypes.byref(dims), int(mask_kind), int(has_sinks), int(dtype),
                            ctypes.byref(pl))
    return st, (pl.as_dict() if st == OK else None)


def nv_sdpa_device_status(stream=0):
    detail = ctypes.c_uint32(0)
    st = lib().nv_sdpa_device_status(stream or None, ctypes.byref(detail))
    return st, detail.value


def nv_sdpa_set_wait_limit(spins: int) -> int:
    return lib().nv_sdpa_set_wait_limit(int(spins))


def nv_sdpa_status_string(status: int) -> str:
    return lib().nv_sdpa_status_string(int(status)).decode()


def nv_sdpa_abi_version() -> int:
    return lib().nv_sdpa_abi_version()


# ----------------------------------------------------------------------------- torch

def _torch_dtype_code(t):
    import torch
    m = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def sdpa(q, k, v, *, mask_kind: str = "none", scale: Optional[float] = None, bool_mask=None,
         sinks=None, out=None, lse=None, want_lse: bool = True, stream=None):
    """Attention forward on CUDA tensors q [B,Hq,Lq,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv].

    Allocates out (and lse, float32) with torch when not given, launches on the current
    torch stream (or `stream`, a torch.cuda.Stream), and returns (out, lse or None).
    """
    import torch
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    B, Hq, Lq, d = q.shape
    Hkv, Lk, dv = k.shape[1], k.shape[2], v.shape[3]
    dt = _torch_dtype_code(q)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, Hq, Lq, dv), dtype=q.dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    mk = MASKS[mask_kind] if isinstance(mask_kind, str) else int(mask_kind)
    if bool_mask is not None and bool_mask.dtype != torch.uint8:
        bool_mask = bool_mask.to(torch.uint8)
    st = (stream or torch.cuda.current_stream(q.device)).cuda_stream
    status = nv_sdpa(q.data_ptr(), k.data_ptr(), v.data_ptr(), (B, Hq, Hkv, Lq, Lk, d, dv), mk,
                     bool_mask.data_ptr() if (bool_mask is not None and mk == 2) else 0,
                     sinks.data_ptr() if sinks is not None else 0, float(scale), out.data_ptr(),
                     lse.data_ptr() if lse is not None else 0, dt, st)
    if status != OK:
        raise NvSdpaError(status)
    return out, lse
