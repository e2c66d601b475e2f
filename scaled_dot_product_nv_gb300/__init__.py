"""Python binding of the nv_sdpa C ABI (include/nv_sdpa.h): argument marshalling only.

Every step of the attention forward runs in the CUDA kernels of libnvsdpa.so; this
module converts Python arguments to C ones and raises on a non-OK status.  There is
no CPU path: if the library is missing, loading it raises.

Raw entry points (same names as the C functions, pointers as ints):
    nv_sdpa, nv_sdpa_ex, nv_sdpa_plan, nv_sdpa_plan_ex, nv_sdpa_paged, nv_sdpa_paged_plan,
    nv_sdpa_host, nv_sdpa_noalloc, nv_sdpa_device_status, nv_sdpa_set_wait_limit,
    nv_sdpa_status_string, nv_sdpa_abi_version
Torch convenience (torch tensors for device memory and the current stream):
    sdpa(q, k, v, mask_kind=..., scale=..., bool_mask=None, sinks=None, window=None,
         add_mask=None)         -- q, k, v, out may be strided views (head dim contiguous)
    sdpa_paged(q, k_cache, v_cache, block_table, seq_lens, mask_kind=..., scale=...,
               sinks=None, window=None)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvsdpa.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
MASKS = {"none": 0, "causal": 1, "bool": 2, "add": 3}
PATHS = {0: "noop", 1: "no_keys", 2: "prefill", 3: "decode"}
KERNELS = {0: "none", 1: "fill", 2: "prefill_tc", 3: "tiled_simt", 4: "decode_mma", 5: "decode_tc"}


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


class Options(ctypes.Structure):
    """nv_sdpa_options: window, additive mask, strides (zero = unused / contiguous)."""
    _fields_ = [("has_window", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("window", ctypes.c_int64), ("add_mask", ctypes.c_void_p),
                ("add_mask_b", ctypes.c_int64), ("add_mask_h", ctypes.c_int64),
                ("q_strides", ctypes.c_int64 * 3), ("k_strides", ctypes.c_int64 * 3),
                ("v_strides", ctypes.c_int64 * 3), ("out_strides", ctypes.c_int64 * 3)]


class PagedDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "Hq", "Hkv", "Lq", "d", "dv", "num_blocks",
                                              "block_size", "max_blocks")]


def make_options(window=None, add_mask=0, add_mask_b=0, add_mask_h=0, q_strides=None,
                 k_strides=None, v_strides=None, out_strides=None) -> Options:
    o = Options()
    if window is not None:
        o.has_window, o.window = 1, int(window)
    o.add_mask = add_mask or None
    o.add_mask_b, o.add_mask_h = int(add_mask_b), int(add_mask_h)
    for name, st in (("q_strides", q_strides), ("k_strides", k_strides), ("v_strides", v_strides),
                     ("out_strides", out_strides)):
        if st is not None:
            getattr(o, name)[:] = [int(x) for x in st]
    return o


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
        L.nv_sdpa_ex.argtypes = sig[:8] + [ctypes.POINTER(Options)] + sig[8:]
        L.nv_sdpa_ex.restype = ctypes.c_int
        L.nv_sdpa_plan_ex.argtypes = [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(Options), ctypes.POINTER(Plan)]
        L.nv_sdpa_plan_ex.restype = ctypes.c_int
        L.nv_sdpa_paged.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(PagedDims), ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int64, vp, ctypes.c_float, vp, vp,
                                    ctypes.c_int, vp]
        L.nv_sdpa_paged.restype = ctypes.c_int
        L.nv_sdpa_paged_plan.argtypes = [ctypes.POINTER(PagedDims), ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(Plan)]
        L.nv_sdpa_paged_plan.restype = ctypes.c_int
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


def nv_sdpa_ex(q, k, v, dims, mask_kind, bool_mask, sinks, scale, options, out, lse, dtype,
               stream) -> int:
    """The C call with options (an Options, or None)."""
    if not isinstance(dims, Dims):
        dims = _dims(*dims)
    return lib().nv_sdpa_ex(q, k, v, ctypes.byref(dims), int(mask_kind), bool_mask or None,
                            sinks or None, ctypes.c_float(scale),
                            ctypes.byref(options) if options is not None else None, out,
                            lse or None, int(dtype), stream or None)


def nv_sdpa_plan_ex(dims, mask_kind, has_sinks, dtype, options=None):
    if not isinstance(dims, Dims):
        dims = _dims(*dims)
    pl = Plan()
    st = lib().nv_sdpa_plan_ex(ctypes.byref(dims), int(mask_kind), int(has_sinks), int(dtype),
                               ctypes.byref(options) if options is not None else None,
                               ctypes.byref(pl))
    return st, (pl.as_dict() if st == OK else None)


def _paged_dims(dims) -> PagedDims:
    return dims if isinstance(dims, PagedDims) else PagedDims(*dims)


def nv_sdpa_paged(q, k_cache, v_cache, block_table, seq_lens, dims, mask_kind, has_window, window,
                  sinks, scale, out, lse, dtype, stream) -> int:
    """The C call; dims a PagedDims or (B, Hq, Hkv, Lq, d, dv, num_blocks, block_size, max_blocks)."""
    return lib().nv_sdpa_paged(q, k_cache, v_cache, block_table, seq_lens,
                               ctypes.byref(_paged_dims(dims)), int(mask_kind), int(has_window),
                               int(window), sinks or None, ctypes.c_float(scale), out, lse or None,
                               int(dtype), stream or None)


def nv_sdpa_paged_plan(dims, mask_kind, has_window, window, has_sinks, dtype):
    pl = Plan()
    st = lib().nv_sdpa_paged_plan(ctypes.byref(_paged_dims(dims)), int(mask_kind), int(has_window),
                                  int(window), int(has_sinks), int(dtype), ctypes.byref(pl))
    return st, (pl.as_dict() if st == OK else None)


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

_TORCH_DTYPE_CODES = None
_RAW_STREAM = None


def _torch_dtype_code(t):
    global _TORCH_DTYPE_CODES
    if _TORCH_DTYPE_CODES is None:
        import torch
        _TORCH_DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    code = _TORCH_DTYPE_CODES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


def _stream_handle(stream, t):
    """The cudaStream_t to launch on: `stream` (a torch.cuda.Stream) if given, else torch's
    current stream on t's device (read without building a Stream object where torch
    exposes the raw handle: the lookup is part of every call's host time)."""
    global _RAW_STREAM
    if stream is not None:
        return stream.cuda_stream
    if _RAW_STREAM is None:
        import torch
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _RAW_STREAM:
        return _RAW_STREAM(t.get_device())
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def _bhl_strides(t):
    """Element strides of a 4-D tensor along [B, H, L]; its last dim must be contiguous."""
    if t.stride(3) != 1 and t.shape[3] > 1:
        raise ValueError("the head dimension must be contiguous")
    return tuple(int(x) for x in t.stride()[:3])


def _strides_or_none(t, contiguous):
    """None (zero strides: the contiguous layout) for a contiguous tensor, else its strides."""
    return None if contiguous else _bhl_strides(t)


def sdpa(q, k, v, *, mask_kind: str = "none", scale: Optional[float] = None, bool_mask=None,
         sinks=None, out=None, lse=None, want_lse: bool = True, stream=None, window=None,
         add_mask=None):
    """Attention forward on CUDA tensors q [B,Hq,Lq,d], k [B,Hkv,Lk,d], v [B,Hkv,Lk,dv].

    q, k, v (and a given out) may be strided views whose last dimension is contiguous
    (transposed [B, L, H, D] layouts, slices of longer caches); they are read in place.
    window: a causal sliding window (mask_kind "causal").  add_mask: the additive mask
    [1|B, 1|Hq, Lq, Lk] of mask_kind "add", in the input dtype.  Allocates out (and lse,
    float32) with torch when not given, launches on the current torch stream (or `stream`,
    a torch.cuda.Stream), and returns (out, lse or None).
    """
    import torch
    for t in (q, k, v):
        if not t.is_cuda:
            raise ValueError("q, k, v must be CUDA tensors")
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
    if lse is not None and not lse.is_contiguous():
        raise ValueError("lse must be contiguous")
    mk = MASKS[mask_kind] if isinstance(mask_kind, str) else int(mask_kind)
    if bool_mask is not None and bool_mask.dtype != torch.uint8:
        bool_mask = bool_mask.to(torch.uint8)
    st = _stream_handle(stream, q)
    cq, ck, cv, co = q.is_contiguous(), k.is_contiguous(), v.is_contiguous(), out.is_contiguous()
    plain = cq and ck and cv and co and window is None and add_mask is None and mk != MASKS["add"]
    if plain:
        status = nv_sdpa(q.data_ptr(), k.data_ptr(), v.data_ptr(), (B, Hq, Hkv, Lq, Lk, d, dv), mk,
                         bool_mask.data_ptr() if (bool_mask is not None and mk == 2) else 0,
                         sinks.data_ptr() if sinks is not None else 0, float(scale), out.data_ptr(),
                         lse.data_ptr() if lse is not None else 0, dt, st)
    else:
        am = 0
        mb = mh = 0
        if add_mask is not None:
            if not add_mask.is_contiguous() or add_mask.dim() != 4:
                raise ValueError("add_mask must be a contiguous [1|B, 1|Hq, Lq, Lk] tensor")
            am, mb, mh = add_mask.data_ptr(), add_mask.shape[0], add_mask.shape[1]
        opts = make_options(window=window, add_mask=am, add_mask_b=mb, add_mask_h=mh,
                            q_strides=_strides_or_none(q, cq), k_strides=_strides_or_none(k, ck),
                            v_strides=_strides_or_none(v, cv), out_strides=_strides_or_none(out, co))
        status = nv_sdpa_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), (B, Hq, Hkv, Lq, Lk, d, dv), mk,
                            bool_mask.data_ptr() if (bool_mask is not None and mk == 2) else 0,
                            sinks.data_ptr() if sinks is not None else 0, float(scale), opts,
                            out.data_ptr(), lse.data_ptr() if lse is not None else 0, dt, st)
    if status != OK:
        raise NvSdpaError(status)
    return out, lse


def sdpa_paged(q, k_cache, v_cache, block_table, seq_lens, *, mask_kind: str = "causal",
               scale: Optional[float] = None, sinks=None, window=None, out=None, lse=None,
               want_lse: bool = True, stream=None):
    """Decode attention over paged caches: q [B,Hq,Lq<=8,d], k_cache [num_blocks,Hkv,bs,d],
    v_cache [num_blocks,Hkv,bs,dv], block_table [B,max_blocks] int32, seq_lens [B] int32
    (all CUDA, contiguous).  Returns (out, lse or None)."""
    import torch
    for t in (q, k_cache, v_cache, block_table, seq_lens):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("paged inputs must be contiguous CUDA tensors")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    B, Hq, Lq, d = q.shape
    nb, Hkv, bs, _ = k_cache.shape
    dv = v_cache.shape[3]
    dt = _torch_dtype_code(q)
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, Hq, Lq, dv), dtype=q.dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    mk = MASKS[mask_kind] if isinstance(mask_kind, str) else int(mask_kind)
    st = _stream_handle(stream, q)
    status = nv_sdpa_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
                           seq_lens.data_ptr(), (B, Hq, Hkv, Lq, d, dv, nb, bs, block_table.shape[1]),
                           mk, window is not None, int(window or 0),
                           sinks.data_ptr() if sinks is not None else 0, float(scale), out.data_ptr(),
                           lse.data_ptr() if lse is not None else 0, dt, st)
    if status != OK:
        raise NvSdpaError(status)
    return out, lse
