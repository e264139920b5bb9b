"""Python binding of libmx, the low-batch MXFP8 block-scaled projection library.

Argument marshalling only: every step runs in the CUDA kernels behind the C ABI
declared in include/mx.h; PyTorch supplies device memory and the current
stream. There is no fallback: if libmx.so is missing or the device is not a
compute-capability 10.3 GPU, the calls raise. Since the C entry points see only
plain pointers, each wrapper first checks every tensor's element type, size,
layout and residency on the handle's GPU (TypeError / ValueError, nothing
launched).

Names and argument order follow the C entry points: mx_create, mx_scale_bytes,
mx_quantize_rows, mx_gemm, mx_gemm_chain, wo_a_grouped, mx_device_status.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmx.so")

MX_OK, MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED, MX_ERR_DEVICE, MX_ERR_CUDA, MX_ERR_TIMEOUT = range(6)
MX_FLAG_PDL = 1

EXPORTS = ["mx_create", "mx_destroy", "mx_scale_bytes", "mx_quantize_rows",
           "mx_rmsnorm_quantize_rows", "mx_gemm", "mx_gemm_bf16", "mx_gemm_chain",
           "mx_gemm_chain_norm", "mx_gemm_chain_noalloc", "wo_a_grouped", "wo_a_grouped_unfused",
           "mx_warmup_bytes", "mx_warmup", "mx_plan_gemm", "mx_plan_chain_push", "mx_device_status",
           "mx_wait_selftest", "mx_status_string"]

_vp, _i, _l, _u = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_uint


class MxWeight(ctypes.Structure):
    _fields_ = [("w", _vp), ("w_scales", _vp), ("n", _i), ("k", _i)]


# reduction forms and push receive areas of the plan queries (include/mx.h)
MX_REDUCE_ITEMS, MX_REDUCE_ROWS, MX_REDUCE_PUSH, MX_REDUCE_PUSH_COMPACT = range(4)
MX_PUSH_NONE, MX_PUSH_COMPACT, MX_PUSH_FULL = range(3)


class MxPlanInfo(ctypes.Structure):
    _fields_ = [("splits", _i), ("stages", _i), ("mtile", _i), ("tmem_cols", _i), ("reduction", _i),
                ("smem", ctypes.c_size_t)]


class MxError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmx.so (built by build.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmx.so is not built ({path}); run mxfp8_block_scaled_06_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.mx_create.argtypes = [ctypes.POINTER(_vp), _i]
    lib.mx_destroy.argtypes = [_vp]
    lib.mx_scale_bytes.argtypes = [_i, _i]
    lib.mx_scale_bytes.restype = ctypes.c_size_t
    lib.mx_quantize_rows.argtypes = [_vp, _i, _i, _vp, _l, _vp, _vp, _i, _vp]
    lib.mx_gemm.argtypes = [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _u, _vp]
    lib.mx_rmsnorm_quantize_rows.argtypes = [_vp, _i, _i, _vp, _l, _vp, ctypes.c_float, _vp, _vp,
                                             _vp, _i, _vp]
    lib.mx_gemm_chain_norm.argtypes = [_vp, _i, _vp, _vp, ctypes.POINTER(MxWeight), _i, _vp,
                                       ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.mx_gemm_bf16.argtypes = [_vp, _i, _i, _i, _vp, _l, _vp, _vp, _vp, _u, _vp]
    lib.mx_gemm_chain.argtypes = [_vp, _i, _vp, _vp, ctypes.POINTER(MxWeight), _i, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp]
    lib.mx_gemm_chain_noalloc.argtypes = [_vp, _i, _vp, _vp, ctypes.POINTER(MxWeight), _i, _vp, _vp]
    lib.mx_warmup_bytes.argtypes = [ctypes.POINTER(MxWeight), _i, ctypes.POINTER(_i), _i]
    lib.mx_warmup_bytes.restype = ctypes.c_size_t
    lib.mx_plan_gemm.argtypes = [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(MxPlanInfo)]
    lib.mx_plan_chain_push.argtypes = [_i, ctypes.POINTER(MxWeight), _i, _i, ctypes.c_size_t, ctypes.c_size_t,
                                       ctypes.POINTER(_i)]
    lib.mx_warmup.argtypes = [_vp, ctypes.POINTER(MxWeight), _i, ctypes.POINTER(_i), _i, _vp,
                              ctypes.c_size_t, _vp]
    lib.wo_a_grouped.argtypes = [_vp, _i, _vp, _l, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i,
                                 _vp, _vp, _vp, _vp, _vp, _i, _vp]
    lib.wo_a_grouped_unfused.argtypes = [_vp, _i, _vp, _l, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i,
                                         _i, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.mx_device_status.argtypes = [_vp, ctypes.POINTER(_i)]
    lib.mx_wait_selftest.argtypes = [_vp, _vp]
    lib.mx_status_string.argtypes = [_i]
    lib.mx_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().mx_status_string(code).decode()


def _check(rc: int, what: str) -> None:
    if rc != MX_OK:
        raise MxError(rc, what)


class Handle:
    """An mx_handle* bound to one device."""

    def __init__(self, ptr: int, device: int):
        self.ptr = ptr
        self.device = device

    def close(self) -> None:
        if self.ptr:
            load_library().mx_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mx_create(device: int = 0) -> Handle:
    p = _vp()
    _check(load_library().mx_create(ctypes.byref(p), device), "mx_create")
    return Handle(p.value, device)


def mx_scale_bytes(rows: int, k: int) -> int:
    return int(load_library().mx_scale_bytes(rows, k))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _empty_u8(shape, device):
    import torch
    return torch.empty(shape, dtype=torch.uint8, device=device)


# The C entry points take plain pointers and cannot see what they point at, so
# the binding checks each tensor before the call: element type, size (so no
# kernel reads or writes past a tensor's end), layout, and that it lives on the
# handle's GPU. Violations raise TypeError / ValueError and launch nothing.
_CODES = _SCALES = _BF16 = None


def _types():
    """(codes, scales, bf16) element types, resolved once."""
    global _CODES, _SCALES, _BF16
    if _CODES is None:
        import torch
        _CODES = (torch.uint8, torch.float8_e4m3fn)
        _SCALES = (torch.uint8,) + ((torch.float8_e8m0fnu,) if hasattr(torch, "float8_e8m0fnu") else ())
        _BF16 = (torch.bfloat16,)
    return _CODES, _SCALES, _BF16


def _codes_types():
    return _types()[0]


def _scale_types():
    return _types()[1]


def _bf16_type():
    return _types()[2]


def _sbytes(rows: int, k: int) -> int:
    """mx_scale_bytes without the library call: ceil128(rows) * ceil4(k / 32), 0 for bad k."""
    if rows < 0 or k <= 0 or k % 32:
        return 0
    return (rows + 127) // 128 * 128 * ((k // 32 + 3) // 4 * 4)


def _resident(h: Handle, host_ok=(), **tensors) -> None:
    """Every given tensor lives on the handle's GPU (checked after all the others,
    so a host tensor is only ever rejected here); those named in host_ok may also
    be pinned host memory, which the kernels address directly (zero-copy)."""
    for name, t in tensors.items():
        if t is None:
            continue
        if name in host_ok and t.device.type == "cpu" and t.is_pinned():
            continue
        if t.get_device() != h.device or not t.is_cuda:
            raise ValueError(f"{name}: on {t.device}, the handle's device is cuda:{h.device}"
                             + (" (or pinned host memory)" if name in host_ok else ""))


def _flat(name: str, t, dtypes, numel: int):
    """A contiguous buffer of one of dtypes holding at least numel elements."""
    if t is None:
        raise ValueError(f"{name}: a tensor is required")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, at least {numel} needed")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def _matrix(name: str, t, dtypes, rows: int, cols: int, row_stride: bool = False):
    """A 2-D tensor of one of dtypes with at least rows rows of exactly cols
    elements; contiguous, or (row_stride) with unit column stride and any row stride."""
    if t is None:
        raise ValueError(f"{name}: a tensor is required")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {dtypes}")
    shape = t.shape
    if len(shape) != 2 or shape[0] < rows or shape[1] != cols:
        raise ValueError(f"{name}: shape {tuple(shape)}, expected [>= {rows}, {cols}]")
    if row_stride:
        st = t.stride()
        if st[1] != 1 or st[0] < cols:
            raise ValueError(f"{name}: layout {st} not supported")
    elif not t.is_contiguous():
        raise ValueError(f"{name}: layout {t.stride()} not supported")
    return t


def _weight(i, w, s):
    if w is None or w.dim() != 2:
        raise ValueError(f"weight {i}: a 2-D [N, K] tensor is required")
    n, k = w.shape
    _matrix(f"weight {i}", w, _codes_types(), n, k)
    _flat(f"weight {i} scales", s, _scale_types(), _sbytes(n, k))
    return n, k


def mx_quantize_rows(h: Handle, x, q=None, scales=None, swizzled: bool = True, stream=None):
    """bf16 [M, K] (row stride x.stride(0)) -> (E4M3 codes uint8 [M, K], scale bytes).
    x may be on the handle's GPU or in pinned host memory (read directly)."""
    import torch
    if x.dim() != 2:
        raise ValueError("x: a 2-D [M, K] tensor is required")
    m, k = x.shape
    _matrix("x", x, (torch.bfloat16,), m, k, row_stride=True)
    sbytes = _sbytes(m, k) if swizzled else m * (k // 32)
    shape = (sbytes,) if swizzled else (m, k // 32)
    if q is not None:
        _matrix("q", q, _codes_types(), m, k)
    if scales is not None:
        _flat("scales", scales, _scale_types(), sbytes)
    if q is None or scales is None:  # outputs to allocate: x must be usable first
        _resident(h, host_ok=("x",), x=x)
    dev = x.device if x.is_cuda else torch.device("cuda", h.device)  # x may be pinned host memory
    q = _empty_u8((m, k), dev) if q is None else q
    scales = _empty_u8(shape, dev) if scales is None else scales
    _resident(h, host_ok=("x",), x=x, q=q, scales=scales)
    _check(load_library().mx_quantize_rows(h.ptr, m, k, _ptr(x), x.stride(0), _ptr(q),
                                           _ptr(scales), int(swizzled), _stream(stream)),
           "mx_quantize_rows")
    return q, scales


def mx_gemm(h: Handle, a, a_scales, w, w_scales, out=None, m: int | None = None,
            pdl: bool = False, stream=None):
    """out[M, N] bf16 = dequant(a[M, K]) x dequant(w[N, K])^T (M = a's rows unless m is given);
    out may be on the handle's GPU or in pinned host memory (written directly)."""
    import torch
    n, k = _weight(0, w, w_scales)
    m = a.shape[0] if m is None else m
    _matrix("a", a, _codes_types(), m, k)
    _flat("a_scales", a_scales, _scale_types(), _sbytes(m, k))
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=w.device)
    _matrix("out", out, (torch.bfloat16,), m, n)
    _resident(h, host_ok=("out",), a=a, a_scales=a_scales, w=w, w_scales=w_scales, out=out)
    _check(load_library().mx_gemm(h.ptr, m, n, k, _ptr(a), _ptr(a_scales), _ptr(w), _ptr(w_scales),
                                  _ptr(out), MX_FLAG_PDL if pdl else 0, _stream(stream)), "mx_gemm")
    return out


def mx_gemm_bf16(h: Handle, x, w, w_scales, out=None, m: int | None = None, pdl: bool = False,
                 stream=None):
    """out[M, N] bf16 = dequant(MXFP8(x[M, K])) x dequant(w[N, K])^T, x bf16 with its
    quantization inside the GEMM kernel (row stride x.stride(0))."""
    import torch
    n, k = _weight(0, w, w_scales)
    m = x.shape[0] if m is None else m
    _matrix("x", x, (torch.bfloat16,), m, k, row_stride=True)
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=w.device)
    _matrix("out", out, (torch.bfloat16,), m, n)
    _resident(h, x=x, w=w, w_scales=w_scales, out=out)
    _check(load_library().mx_gemm_bf16(h.ptr, m, n, k, _ptr(x), x.stride(0), _ptr(w), _ptr(w_scales),
                                       _ptr(out), MX_FLAG_PDL if pdl else 0, _stream(stream)),
           "mx_gemm_bf16")
    return out


def _chain_buffers(a1, a1_scales, weights, g1_cols, a2, a2_scales, a3, a3_scales, out):
    """Checks and allocations shared by the two chain entry points."""
    import torch
    if len(weights) != 3:
        raise ValueError("weights: three (w, w_scales) pairs are required")
    (n1, k1), (n2, _), (n3, _) = (_weight(i, w, s) for i, (w, s) in enumerate(weights))
    m = a1.shape[0]
    dev = a1.device
    _matrix("a1", a1, _codes_types(), m, k1)
    _flat("a1_scales", a1_scales, _scale_types(), _sbytes(m, k1))
    a2 = _empty_u8((m, g1_cols), dev) if a2 is None else _matrix("a2", a2, _codes_types(), m, g1_cols)
    a2_scales = (_empty_u8((_sbytes(m, g1_cols),), dev) if a2_scales is None else
                 _flat("a2_scales", a2_scales, _scale_types(), _sbytes(m, g1_cols)))
    a3 = _empty_u8((m, n2), dev) if a3 is None else _matrix("a3", a3, _codes_types(), m, n2)
    a3_scales = (_empty_u8((_sbytes(m, n2),), dev) if a3_scales is None else
                 _flat("a3_scales", a3_scales, _scale_types(), _sbytes(m, n2)))
    out = torch.empty((m, n3), dtype=torch.bfloat16, device=dev) if out is None else out
    _matrix("out", out, (torch.bfloat16,), m, n3)
    ws = (MxWeight * 3)(*[MxWeight(_ptr(w), _ptr(s), w.shape[0], w.shape[1]) for w, s in weights])
    return m, dev, ws, (n1, n2, n3), a2, a2_scales, a3, a3_scales, out


def _chain_resident(h: Handle, a1, a1_scales, weights, a2, a2_scales, a3, a3_scales, out):
    _resident(h, a1=a1, a1_scales=a1_scales, a2=a2, a2_scales=a2_scales, a3=a3, a3_scales=a3_scales,
              out=out, **{f"weight {i}": w for i, (w, _) in enumerate(weights)},
              **{f"weight {i} scales": s for i, (_, s) in enumerate(weights)})


def mx_gemm_chain(h: Handle, a1, a1_scales, weights, g1_cols: int = 1536, out=None,
                  a2=None, a2_scales=None, a3=None, a3_scales=None, debug: bool = False,
                  stream=None) -> dict:
    """Three projections on one stream with PDL: G1 -> MXFP8 requant of its first
    g1_cols columns -> G2 -> requant -> G3. weights = [(w, w_scales)] * 3."""
    import torch
    m, dev, ws, (n1, n2, n3), a2, a2_scales, a3, a3_scales, out = _chain_buffers(
        a1, a1_scales, weights, g1_cols, a2, a2_scales, a3, a3_scales, out)
    d1 = torch.empty((m, n1), dtype=torch.bfloat16, device=dev) if debug else None
    d2 = torch.empty((m, n2), dtype=torch.bfloat16, device=dev) if debug else None
    _chain_resident(h, a1, a1_scales, weights, a2, a2_scales, a3, a3_scales, out)
    _check(load_library().mx_gemm_chain(h.ptr, m, _ptr(a1), _ptr(a1_scales), ws, g1_cols, _ptr(a2),
                                        _ptr(a2_scales), _ptr(a3), _ptr(a3_scales), _ptr(out),
                                        _ptr(d1), _ptr(d2), _stream(stream)), "mx_gemm_chain")
    return dict(out=out, a2=a2, a2_scales=a2_scales, a3=a3, a3_scales=a3_scales, out1=d1, out2=d2)


def mx_gemm_chain_noalloc(h: Handle, a1, a1_scales, weights, g1_cols: int = 1536, out=None,
                          stream=None):
    """The chain for callers that cannot allocate device memory: only the inputs
    and the output are passed; the library keeps the two intermediates in a fixed
    1 MiB device array (see include/mx.h). Raises MxError (MX_ERR_UNSUPPORTED)
    when the intermediates do not fit; calls that overlap on the GPU race."""
    import torch
    if len(weights) != 3:
        raise ValueError("weights: three (w, w_scales) pairs are required")
    (_, k1), _, (n3, _) = (_weight(i, w, s) for i, (w, s) in enumerate(weights))
    m = a1.shape[0]
    _matrix("a1", a1, _codes_types(), m, k1)
    _flat("a1_scales", a1_scales, _scale_types(), _sbytes(m, k1))
    out = torch.empty((m, n3), dtype=torch.bfloat16, device=a1.device) if out is None else out
    _matrix("out", out, (torch.bfloat16,), m, n3)
    ws = (MxWeight * 3)(*[MxWeight(_ptr(w), _ptr(s), w.shape[0], w.shape[1]) for w, s in weights])
    _resident(h, a1=a1, a1_scales=a1_scales, out=out,
              **{f"weight {i}": w for i, (w, _) in enumerate(weights)},
              **{f"weight {i} scales": s for i, (_, s) in enumerate(weights)})
    _check(load_library().mx_gemm_chain_noalloc(h.ptr, m, _ptr(a1), _ptr(a1_scales), ws, g1_cols,
                                                _ptr(out), _stream(stream)),
           "mx_gemm_chain_noalloc (the intermediates must fit in the library's 1 MiB array)")
    return out


def mx_rmsnorm_quantize_rows(h: Handle, x, norm_weight, eps: float, q=None, scales=None,
                             swizzled: bool = True, y: bool = False, stream=None):
    """bf16 [M, K] (row stride x.stride(0)) -> RMS-normalized with norm_weight [K] bf16 and
    eps, rounded to bf16 (returned as y when asked) and MX-quantized: (q, scales, y)."""
    import torch
    if x.dim() != 2:
        raise ValueError("x: a 2-D [M, K] tensor is required")
    m, k = x.shape
    _matrix("x", x, (torch.bfloat16,), m, k, row_stride=True)
    _flat("norm_weight", norm_weight, (torch.bfloat16,), k)
    sbytes = _sbytes(m, k) if swizzled else m * (k // 32)
    q = _empty_u8((m, k), x.device) if q is None else _matrix("q", q, _codes_types(), m, k)
    shape = (sbytes,) if swizzled else (m, k // 32)
    scales = _empty_u8(shape, x.device) if scales is None else _flat("scales", scales, _scale_types(), sbytes)
    yt = torch.empty((m, k), dtype=torch.bfloat16, device=x.device) if y else None
    _resident(h, x=x, norm_weight=norm_weight, q=q, scales=scales)
    _check(load_library().mx_rmsnorm_quantize_rows(h.ptr, m, k, _ptr(x), x.stride(0),
                                                   _ptr(norm_weight), float(eps), _ptr(yt), _ptr(q),
                                                   _ptr(scales), int(swizzled), _stream(stream)),
           "mx_rmsnorm_quantize_rows")
    return q, scales, yt


def mx_gemm_chain_norm(h: Handle, a1, a1_scales, weights, norm_weight, eps: float,
                       g1_cols: int = 1536, out=None, out1=None, a2=None, a2_scales=None, a3=None,
                       a3_scales=None, debug: bool = False, stream=None) -> dict:
    """mx_gemm_chain with the RMS-norm split between G1 and G2: G1's bf16 output goes
    to out1 (qr | kv), qr is normalized and quantized for G2."""
    import torch
    m, dev, ws, (n1, n2, n3), a2, a2_scales, a3, a3_scales, out = _chain_buffers(
        a1, a1_scales, weights, g1_cols, a2, a2_scales, a3, a3_scales, out)
    _flat("norm_weight", norm_weight, (torch.bfloat16,), g1_cols)
    out1 = torch.empty((m, n1), dtype=torch.bfloat16, device=dev) if out1 is None else out1
    _matrix("out1", out1, (torch.bfloat16,), m, n1)
    dy = torch.empty((m, g1_cols), dtype=torch.bfloat16, device=dev) if debug else None
    d2 = torch.empty((m, n2), dtype=torch.bfloat16, device=dev) if debug else None
    _chain_resident(h, a1, a1_scales, weights, a2, a2_scales, a3, a3_scales, out)
    _resident(h, norm_weight=norm_weight, out1=out1)
    _check(load_library().mx_gemm_chain_norm(h.ptr, m, _ptr(a1), _ptr(a1_scales), ws, g1_cols,
                                             _ptr(norm_weight), float(eps), _ptr(out1), _ptr(a2),
                                             _ptr(a2_scales), _ptr(a3), _ptr(a3_scales), _ptr(out),
                                             _ptr(dy), _ptr(d2), _stream(stream)),
           "mx_gemm_chain_norm")
    return dict(out=out, out1=out1, a2=a2, a2_scales=a2_scales, a3=a3, a3_scales=a3_scales, y=dy,
                out2=d2)


def _wo_a_inputs(x, positions, cos_sin, w, w_scales, n_groups, heads_per_group,
                 o_lora_rank, d_nope, d_rope):
    """Checks shared by the two WO-A entry points; returns (T, K of all groups, columns)."""
    import torch
    t = x.shape[0]
    kall = n_groups * heads_per_group * (d_nope + d_rope)
    cols = n_groups * o_lora_rank
    if x.dtype != torch.bfloat16:
        raise TypeError(f"x: dtype {x.dtype}, expected torch.bfloat16")
    # each token's heads x dims are contiguous; tokens are x.stride(0) elements apart
    if x.dim() < 2 or x.stride(-1) != 1 or not x[0].is_contiguous() or x[0].numel() != kall:
        raise ValueError(f"x: each token must hold {kall} contiguous elements")
    if x.stride(0) < kall:
        raise ValueError(f"x: token stride {x.stride(0)} below {kall}")
    _flat("positions", positions, (torch.int64,), t)
    if cos_sin.dim() != 2 or cos_sin.shape[1] != d_rope:
        raise ValueError(f"cos_sin: shape {tuple(cos_sin.shape)}, expected [max_pos, {d_rope}]")
    _flat("cos_sin", cos_sin, (torch.float32,), 0)
    _matrix("w", w, _codes_types(), cols, heads_per_group * (d_nope + d_rope))
    _flat("w_scales", w_scales, _scale_types(), _sbytes(cols, heads_per_group * (d_nope + d_rope)))
    return t, kall, cols


def _wo_a_resident(h: Handle, x, positions, cos_sin, w, w_scales):
    _resident(h, x=x, positions=positions, cos_sin=cos_sin, w=w, w_scales=w_scales)


def wo_a_grouped(h: Handle, x, positions, cos_sin, w, w_scales, n_groups: int,
                 heads_per_group: int, o_lora_rank: int, d_nope: int = 448, d_rope: int = 64,
                 q=None, q_scales=None, debug: bool = False, early_trigger: bool = False,
                 z: bool = False, stream=None) -> dict:
    """x: bf16 [T, heads, d_nope + d_rope] (token stride x.stride(0)); returns the
    MXFP8 activation (q, q_scales) for wo_b, plus debug tensors if asked: z (bf16
    before requantization) with z or debug, the quantized activation with debug
    (which keeps the call on the fused kernel at every T)."""
    import torch
    t, kall, cols = _wo_a_inputs(x, positions, cos_sin, w, w_scales, n_groups, heads_per_group,
                                 o_lora_rank, d_nope, d_rope)
    dev = x.device
    q = _empty_u8((t, cols), dev) if q is None else _matrix("q", q, _codes_types(), t, cols)
    q_scales = (_empty_u8((_sbytes(t, cols),), dev) if q_scales is None else
                _flat("q_scales", q_scales, _scale_types(), _sbytes(t, cols)))
    dz = torch.empty((t, cols), dtype=torch.bfloat16, device=dev) if debug or z else None
    dxq = _empty_u8((t, kall), dev) if debug else None
    dxs = _empty_u8((t, kall // 32), dev) if debug else None
    _wo_a_resident(h, x, positions, cos_sin, w, w_scales)
    _resident(h, q=q, q_scales=q_scales)
    _check(load_library().wo_a_grouped(h.ptr, t, _ptr(x), x.stride(0), _ptr(positions),
                                       _ptr(cos_sin), cos_sin.shape[0], _ptr(w), _ptr(w_scales),
                                       n_groups, heads_per_group, d_nope, d_rope, o_lora_rank,
                                       _ptr(q), _ptr(q_scales), _ptr(dz), _ptr(dxq), _ptr(dxs),
                                       int(early_trigger), _stream(stream)), "wo_a_grouped")
    return dict(q=q, q_scales=q_scales, z=dz, xq=dxq, xs=dxs)


def wo_a_grouped_unfused(h: Handle, x, positions, cos_sin, w, w_scales, n_groups: int,
                         heads_per_group: int, o_lora_rank: int, d_nope: int = 448,
                         d_rope: int = 64, q=None, q_scales=None, xq=None, xq_scales=None,
                         z: bool = False, stream=None) -> dict:
    """wo_a_grouped in two launches (RoPE + quantize into the caller-owned xq, then a
    grouped GEMM with the requantization fused); for token counts up to 256."""
    import torch
    t, kall, cols = _wo_a_inputs(x, positions, cos_sin, w, w_scales, n_groups, heads_per_group,
                                 o_lora_rank, d_nope, d_rope)
    dev = x.device
    q = _empty_u8((t, cols), dev) if q is None else _matrix("q", q, _codes_types(), t, cols)
    q_scales = (_empty_u8((_sbytes(t, cols),), dev) if q_scales is None else
                _flat("q_scales", q_scales, _scale_types(), _sbytes(t, cols)))
    xq = _empty_u8((t, kall), dev) if xq is None else _matrix("xq", xq, _codes_types(), t, kall)
    xq_scales = (_empty_u8((_sbytes(t, kall),), dev) if xq_scales is None else
                 _flat("xq_scales", xq_scales, _scale_types(), _sbytes(t, kall)))
    zt = torch.empty((t, cols), dtype=torch.bfloat16, device=dev) if z else None
    _wo_a_resident(h, x, positions, cos_sin, w, w_scales)
    _resident(h, q=q, q_scales=q_scales, xq=xq, xq_scales=xq_scales)
    _check(load_library().wo_a_grouped_unfused(h.ptr, t, _ptr(x), x.stride(0), _ptr(positions),
                                               _ptr(cos_sin), cos_sin.shape[0], _ptr(w),
                                               _ptr(w_scales), n_groups, heads_per_group, d_nope,
                                               d_rope, o_lora_rank, _ptr(xq), _ptr(xq_scales),
                                               _ptr(zt), _ptr(q), _ptr(q_scales), _stream(stream)),
           "wo_a_grouped_unfused")
    return dict(q=q, q_scales=q_scales, z=zt, xq=xq, xq_scales=xq_scales)


def mx_warmup(h: Handle, weights, rows, stream=None) -> list:
    """Ready the GEMM of every distinct weight shape at each row count (plans,
    tensor maps, one launch on a zero MXFP8 activation). weights: (w, w_scales)
    pairs; returns the runs' bf16 outputs ([rows, n], all zero for finite
    weights) in run order: shapes in increasing (n, k), then rows as given."""
    import torch
    if not weights or not rows:
        raise ValueError("mx_warmup needs at least one weight and one row count")
    ws = (MxWeight * len(weights))(*[MxWeight(_ptr(w), _ptr(s), w.shape[0], w.shape[1])
                                     for w, s in weights])
    rr = (_i * len(rows))(*[int(r) for r in rows])
    lib = load_library()
    nbytes = int(lib.mx_warmup_bytes(ws, len(weights), rr, len(rows)))
    if nbytes == 0:
        raise MxError(MX_ERR_INVALID_ARG, "mx_warmup_bytes")
    dev = weights[0][0].device
    scratch = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
    off0 = (-scratch.data_ptr()) % 256
    buf = scratch[off0:off0 + nbytes]
    _check(lib.mx_warmup(h.ptr, ws, len(weights), rr, len(rows), _ptr(buf), nbytes, _stream(stream)),
           "mx_warmup")
    shapes = sorted({(w.shape[0], w.shape[1]) for w, _ in weights})
    r256 = lambda v: (v + 255) // 256 * 256
    off = r256(max(r * k for _, k in shapes for r in rows)) + \
        r256(max(mx_scale_bytes(r, k) for _, k in shapes for r in rows))
    outs = []
    for n, k in shapes:
        for r in rows:
            outs.append(buf[off:off + r * n * 2].view(torch.bfloat16).view(r, n))
            off += r256(r * n * 2)
    return outs


def mx_plan_gemm(m: int, n: int, k: int, sm_count: int = 152, fused: bool = False, norm: bool = False,
                 push: int = MX_PUSH_FULL) -> dict:
    """The launch plan mx_gemm (fused: mx_gemm_bf16; norm: the chain-norm's
    G2) makes for [m, k] x [n, k]^T on a device with sm_count SMs. Host only."""
    info = MxPlanInfo()
    _check(load_library().mx_plan_gemm(m, n, k, sm_count, int(fused), int(norm), push, ctypes.byref(info)),
           "mx_plan_gemm")
    return {f: getattr(info, f) for f, _ in MxPlanInfo._fields_}


def mx_plan_chain_push(m: int, shapes, norm: bool = False, sm_count: int = 152, smem_per_sm: int = 233472,
                       smem_reserved: int = 1024) -> list:
    """The push receive area (MX_PUSH_*) of each projection of mx_gemm_chain
    (norm: mx_gemm_chain_norm) at m rows; shapes = [(n, k)] * 3. Host only."""
    ws = (MxWeight * 3)(*[MxWeight(None, None, n, k) for n, k in shapes])
    modes = (_i * 3)()
    _check(load_library().mx_plan_chain_push(m, ws, int(norm), sm_count, smem_per_sm, smem_reserved, modes),
           "mx_plan_chain_push")
    return list(modes)


def mx_device_status(h: Handle) -> int:
    """MX_OK, or the error a kernel recorded since the last call (synchronizes)."""
    v = _i(0)
    _check(load_library().mx_device_status(h.ptr, ctypes.byref(v)), "mx_device_status")
    return v.value


def mx_wait_selftest(h: Handle, stream=None) -> None:
    """Launch the bounded-wait diagnostic: about one second later the kernel gives
    up on a barrier nothing completes, and the next mx_device_status reports
    MX_ERR_TIMEOUT."""
    _check(load_library().mx_wait_selftest(h.ptr, _stream(stream)), "mx_wait_selftest")
