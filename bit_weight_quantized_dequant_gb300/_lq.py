"""ctypes binding of the liblq C ABI (include/lq.h).

Tensors are PyTorch CUDA tensors; only their device pointers, the current CUDA
stream and plain sizes cross the boundary.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from pathlib import Path

LQ_OK, LQ_ERR_INVALID_ARG, LQ_ERR_UNSUPPORTED, LQ_ERR_ALIGNMENT, LQ_ERR_WORKSPACE, LQ_ERR_CUDA, LQ_ERR_TIMEOUT, \
    LQ_ERR_RANGE = range(8)
FMT_2BIT, FMT_NF4, FMT_INT4, FMT_NF4_DQ = 1, 2, 3, 4
F32, F16, BF16 = 0, 1, 2

#: every entry point include/lq.h declares
EXPORTED = ("lq_create", "lq_destroy", "lq_status_string", "lq_sync", "lq_dequant", "lq_gemv",
            "lq_anchor_count",
            "lq_gemv_grouped", "lq_gemv_layers", "lq_gemm", "lq_gemm_grouped", "lq_gemv_noalloc",
            "lq_select_anchors", "lq_quantize_2bit", "lq_quantize_nf4",
            "lq_stream_create", "lq_stream_run", "lq_stream_destroy", "lq_stream_run_direct",
            "lq_selftest_wait")

_LIB = None


class LQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _LIB.lq_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class lq_problem(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int), ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
        ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
        ("anchor_idx", ctypes.c_void_p), ("anchor_w", ctypes.c_void_p),
        ("A", ctypes.c_int), ("ld_anchor", ctypes.c_int),
        ("x", ctypes.c_void_p), ("x_dtype", ctypes.c_int), ("y", ctypes.c_void_p), ("y_dtype", ctypes.c_int),
        ("batch", ctypes.c_int),
        ("stride_codes", ctypes.c_int64), ("stride_scales", ctypes.c_int64), ("stride_offsets", ctypes.c_int64),
        ("stride_anchor_idx", ctypes.c_int64), ("stride_anchor_w", ctypes.c_int64),
        ("stride_x", ctypes.c_int64), ("stride_y", ctypes.c_int64),
    ]


def library_path() -> Path:
    from .build import LIB
    return LIB


def load_library(build_if_missing: bool = True):
    """Load liblq.so (building it first if asked and needed); raises if it cannot be loaded."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if build_if_missing:
        from .build import build
        path = build()
    if not path.exists():
        raise RuntimeError(f"liblq.so not built at {path}; run bit_weight_quantized_dequant_gb300.build()")
    L = ctypes.CDLL(str(path))
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.lq_create.argtypes = [ctypes.POINTER(P), I, S]
    L.lq_create.restype = I
    L.lq_destroy.argtypes = [P]
    L.lq_destroy.restype = I
    L.lq_sync.argtypes = [P]
    L.lq_sync.restype = I
    L.lq_status_string.argtypes = [I]
    L.lq_status_string.restype = ctypes.c_char_p
    L.lq_dequant.argtypes = [P, I, P, P, P, P, P, I, I, P, I, I, I, P]
    L.lq_dequant.restype = I
    L.lq_gemv.argtypes = [P, I, P, P, P, P, P, I, I, P, I, P, I, I, I, I, P]
    L.lq_gemv.restype = I
    L.lq_gemm.argtypes = [P, I, P, P, P, P, P, I, I, P, I, P, I, I, I, I, P]
    L.lq_gemm.restype = I
    L.lq_gemv_noalloc.argtypes = [I, P, P, P, P, P, I, I, P, I, P, I, I, I, I, P]
    L.lq_gemv_noalloc.restype = I
    L.lq_gemv_grouped.argtypes = [P, ctypes.POINTER(lq_problem), I, P]
    L.lq_gemv_grouped.restype = I
    L.lq_gemv_layers.argtypes = [P, ctypes.POINTER(lq_problem), ctypes.POINTER(I), I, P]
    L.lq_gemv_layers.restype = I
    L.lq_gemm_grouped.argtypes = [P, ctypes.POINTER(lq_problem), I, P]
    L.lq_gemm_grouped.restype = I
    L.lq_anchor_count.argtypes = [I]
    L.lq_anchor_count.restype = I
    L.lq_select_anchors.argtypes = [P, P, I, I, P, I, P, P]
    L.lq_select_anchors.restype = I
    L.lq_quantize_2bit.argtypes = [P, P, I, I, P, I, P, P, P, P, I, P]
    L.lq_quantize_2bit.restype = I
    L.lq_quantize_nf4.argtypes = [P, P, I, I, P, P, P]
    L.lq_quantize_nf4.restype = I
    L.lq_stream_create.argtypes = [ctypes.POINTER(P), P, S]
    L.lq_stream_create.restype = I
    L.lq_stream_run.argtypes = [P, P, S, S, I, ctypes.POINTER(lq_problem), I, ctypes.c_int64, P]
    L.lq_stream_run.restype = I
    L.lq_stream_destroy.argtypes = [P]
    L.lq_stream_destroy.restype = I
    L.lq_stream_run_direct.argtypes = [P, P, S, S, I, ctypes.POINTER(lq_problem), I, ctypes.c_int64, P]
    L.lq_stream_run_direct.restype = I
    L.lq_selftest_wait.argtypes = [P, ctypes.c_uint, P]
    L.lq_selftest_wait.restype = I
    _LIB = L
    return L


def exported_symbols(path: Path | None = None) -> list[str]:
    """Names from EXPORTED that the library resolves (no GPU needed)."""
    L = ctypes.CDLL(str(path or library_path()))
    return [n for n in EXPORTED if hasattr(L, n)]


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[t.dtype]


def _stream(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream) or None


@dataclass
class QuantWeights:
    """One quantized matrix W [N][K] in device memory (layouts as in include/lq.h)."""
    format: int
    N: int
    K: int
    codes: object                 # uint8 tensor
    scales: object                # float16 [N][K/32] (2-bit, INT4), float32 [N][K/64] (NF4) or uint8 [N][K/64] (NF4-DQ)
    offsets: object = None        # float16 [N][K/32] (2-bit), int32 permutation [K] (INT4) or float32 second level (NF4-DQ)
    anchor_idx: object = None     # int32 [A]
    anchor_w: object = None       # float16 [N][ld_anchor]
    A: int = 0
    ld_anchor: int = 0

    @staticmethod
    def from_host(packed: dict, fmt: int, device="cuda") -> "QuantWeights":
        """Copy a packed host dict (numpy arrays, bit patterns as uint16) to the device."""
        import numpy as np
        import torch

        def t(a, dtype):
            return torch.from_numpy(np.ascontiguousarray(a)).view(dtype).to(device)
        if fmt in (FMT_2BIT, FMT_INT4):
            A = int(packed["A"])
            off = t(packed["offsets"], torch.float16) if fmt == FMT_2BIT else t(packed["perm"], torch.int32)
            return QuantWeights(fmt, int(packed["N"]), int(packed["K"]), t(packed["codes"], torch.uint8),
                                t(packed["scales"], torch.float16), off,
                                t(packed["anchor_idx"], torch.int32) if A > 0 else None,
                                t(packed["anchor_w"], torch.float16) if A > 0 else None, A, int(packed["ld_anchor"]))
        if fmt == FMT_NF4_DQ:
            return QuantWeights(FMT_NF4_DQ, int(packed["N"]), int(packed["K"]), t(packed["codes"], torch.uint8),
                                t(packed["acodes"], torch.uint8), t(packed["second"], torch.float32))
        return QuantWeights(FMT_NF4, int(packed["N"]), int(packed["K"]), t(packed["codes"], torch.uint8),
                            t(packed["absmax"], torch.float32))

    def args(self):
        return (self.format, _ptr(self.codes), _ptr(self.scales), _ptr(self.offsets), _ptr(self.anchor_idx),
                _ptr(self.anchor_w), int(self.A), int(self.ld_anchor))


class Handle:
    """An lq handle on one CUDA device, with its split-K workspace."""

    def __init__(self, device: int = 0, workspace_bytes: int = 0):
        self._lib = load_library()
        h = ctypes.c_void_p()
        st = self._lib.lq_create(ctypes.byref(h), int(device), int(workspace_bytes))
        if st != LQ_OK:
            raise LQError(st, "lq_create")
        self._h = h
        self.device = device

    def close(self):
        if getattr(self, "_h", None):
            st = self._lib.lq_destroy(self._h)
            self._h = None
            if st != LQ_OK:
                raise LQError(st, "lq_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def raw(self):
        return self._h

    def sync(self):
        st = self._lib.lq_sync(self._h)
        if st != LQ_OK:
            raise LQError(st, "lq_sync")

    def dequant(self, w: QuantWeights, out=None, out_dtype=None, stream=None):
        import torch
        if out is None:
            out = torch.empty((w.N, w.K), dtype=out_dtype or torch.float32, device=w.codes.device)
        fmt, c, s, o, ai, aw, A, ld = w.args()
        st = self._lib.lq_dequant(self._h, fmt, c, s, o, ai, aw, A, ld, _ptr(out), _dtype_code(out), w.N, w.K,
                                  _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_dequant")
        return out

    def _mm(self, fn, name, w: QuantWeights, x, y=None, y_dtype=None, stream=None):
        import torch
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, w.N), dtype=y_dtype or torch.float32, device=x.device)
        fmt, c, s, o, ai, aw, A, ld = w.args()
        st = fn(self._h, fmt, c, s, o, ai, aw, A, ld, _ptr(x), _dtype_code(x), _ptr(y), _dtype_code(y), M, w.N, w.K,
                _stream(stream))
        if st != LQ_OK:
            raise LQError(st, name)
        return y

    def gemv(self, w: QuantWeights, x, y=None, y_dtype=None, stream=None):
        """y = x * W_eff^T for 1 <= M <= 32 tokens (decode)."""
        return self._mm(self._lib.lq_gemv, "lq_gemv", w, x, y, y_dtype, stream)

    def gemm(self, w: QuantWeights, x, y=None, y_dtype=None, stream=None):
        """y = x * W_eff^T on the tcgen05 tensor-core path (prefill)."""
        return self._mm(self._lib.lq_gemm, "lq_gemm", w, x, y, y_dtype, stream)

    @staticmethod
    def problem(w: QuantWeights, x, y, batch: int = 1, strides: dict | None = None) -> lq_problem:
        """Describe one (batched) product for gemv_grouped; strides are in bytes."""
        p = lq_problem()
        fmt, c, s, o, ai, aw, A, ld = w.args()
        p.format, p.M, p.N, p.K = fmt, int(x.shape[-2]), w.N, w.K
        p.codes, p.scales, p.offsets, p.anchor_idx, p.anchor_w = c, s, o, ai, aw
        p.A, p.ld_anchor = A, ld
        p.x, p.x_dtype, p.y, p.y_dtype = _ptr(x), _dtype_code(x), _ptr(y), _dtype_code(y)
        p.batch = int(batch)
        for k, v in (strides or {}).items():
            setattr(p, "stride_" + k, int(v))
        return p

    @staticmethod
    def prepare(problems):
        """The C array of a list of problems, built once: a decode loop passes it to gemv_grouped
        every token instead of the list (no per-call marshalling)."""
        return (lq_problem * len(problems))(*problems)

    def gemv_grouped(self, problems, stream=None):
        arr = problems if isinstance(problems, ctypes.Array) else (lq_problem * len(problems))(*problems)
        st = self._lib.lq_gemv_grouped(self._h, arr, len(arr), _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_gemv_grouped")

    def gemv_layers(self, layers, stream=None):
        """Consecutive layers (each a list of problems) in one call; a layer may read what the
        layers before it wrote."""
        flat = [p for layer in layers for p in layer]
        arr = (lq_problem * len(flat))(*flat)
        counts = (ctypes.c_int * len(layers))(*[len(layer) for layer in layers])
        st = self._lib.lq_gemv_layers(self._h, arr, counts, len(layers), _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_gemv_layers")

    def selftest_wait(self, limit_us: int, stream=None):
        """Run the bounded-wait self-test: a wait that nothing completes gives up after
        limit_us; the next sync() raises LQError with status LQ_ERR_TIMEOUT."""
        st = self._lib.lq_selftest_wait(self._h, int(limit_us), _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_selftest_wait")

    # ---- quantizers (the converter step; include/lq.h gives the definitions) ----

    @staticmethod
    def _weights_arg(W):
        import torch
        if W.dtype != torch.float32 or W.dim() != 2 or not W.is_contiguous() or not W.is_cuda:
            raise ValueError("W must be a contiguous fp32 [N][K] CUDA tensor")
        return W.shape[0], W.shape[1]

    def select_anchors(self, W, A=None, profile=None, stream=None):
        """Anchor columns of W: the A largest ||W[:,c]||_2 * profile_c (ties to the lower
        column), ascending, as an int32 CUDA tensor.  A defaults to the library's
        outlier-anchor count for K (lq_anchor_count); profile is an fp64 [K] CUDA tensor
        (None: all ones)."""
        import torch
        N, K = self._weights_arg(W)
        A = self._lib.lq_anchor_count(K) if A is None else int(A)
        idx = torch.empty(max(A, 0), dtype=torch.int32, device=W.device)
        if profile is not None and (profile.dtype != torch.float64 or profile.numel() != K or not profile.is_contiguous()):
            raise ValueError("profile must be a contiguous fp64 [K] tensor")
        st = self._lib.lq_select_anchors(self._h, _ptr(W), N, K, _ptr(profile), A, _ptr(idx) if A > 0 else None,
                                         _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_select_anchors")
        return idx

    def quantize_2bit(self, W, anchor_idx=None, ld_anchor=None, stream=None) -> QuantWeights:
        """The 2-bit Lloyd-Max G=32 quantizer of W (fp32 [N][K] on the device), with the given
        anchor columns (int32 CUDA tensor, ascending) kept in binary16."""
        import torch
        N, K = self._weights_arg(W)
        A = 0 if anchor_idx is None else int(anchor_idx.numel())
        ld = (int(ld_anchor) if ld_anchor is not None else max(8, (A + 7) // 8 * 8)) if A > 0 else 0
        dev = W.device
        codes = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
        scales = torch.empty((N, K // 32), dtype=torch.float16, device=dev)
        offsets = torch.empty((N, K // 32), dtype=torch.float16, device=dev)
        anchor_w = torch.empty((N, ld), dtype=torch.float16, device=dev) if A > 0 else None
        st = self._lib.lq_quantize_2bit(self._h, _ptr(W), N, K, _ptr(anchor_idx) if A > 0 else None, A, _ptr(codes),
                                        _ptr(scales), _ptr(offsets), _ptr(anchor_w), ld, _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_quantize_2bit")
        return QuantWeights(FMT_2BIT, N, K, codes, scales, offsets, anchor_idx if A > 0 else None, anchor_w, A, ld)

    def quantize_nf4(self, W, stream=None) -> QuantWeights:
        """The NF4 block-64 quantizer of W (fp32 [N][K] on the device)."""
        import torch
        N, K = self._weights_arg(W)
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
        absmax = torch.empty((N, max(K // 64, 1)), dtype=torch.float32, device=W.device)
        st = self._lib.lq_quantize_nf4(self._h, _ptr(W), N, K, _ptr(codes), _ptr(absmax), _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_quantize_nf4")
        return QuantWeights(FMT_NF4, N, K, codes, absmax)

    def gemm_grouped(self, problems, stream=None):
        """Several prefill products (same format and x dtype) in one tensor-core launch."""
        arr = (lq_problem * len(problems))(*problems)
        st = self._lib.lq_gemm_grouped(self._h, arr, len(problems), _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_gemm_grouped")


# ---- layer streaming (weights in host memory, two device slots) --------------------

def pack_layer(packed: list, fmt: int, align: int = 256):
    """Lay one layer's packed host dicts (the layout of QuantWeights.from_host) out as one
    byte blob.  Returns (blob as uint8 numpy array, per-matrix dict of byte offsets)."""
    import numpy as np
    parts, offs = [], []
    pos = 0

    def add(a):
        nonlocal pos
        b = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        pad = (-pos) % align
        if pad:
            parts.append(np.zeros(pad, np.uint8))
            pos += pad
        o = pos
        parts.append(b)
        pos += b.nbytes
        return o

    for p in packed:
        d = {"codes": add(p["codes"]), "N": int(p["N"]), "K": int(p["K"]), "A": 0, "ld_anchor": 0}
        if fmt == FMT_2BIT:
            d["scales"] = add(p["scales"])
            d["offsets"] = add(p["offsets"])
            A = int(p["A"])
            d["A"], d["ld_anchor"] = A, (int(p["ld_anchor"]) if A > 0 else 0)
            d["anchor_idx"] = add(p["anchor_idx"]) if A > 0 else 0
            d["anchor_w"] = add(p["anchor_w"]) if A > 0 else 0
        else:
            d["scales"] = add(p["absmax"])
            d["offsets"] = d["anchor_idx"] = d["anchor_w"] = 0
        offs.append(d)
    pad = (-pos) % align
    if pad:
        parts.append(np.zeros(pad, np.uint8))
    return np.concatenate(parts), offs


class LayerStream:
    """A decode pass over a layer stack whose packed weights live in (pinned) host memory:
    layer l+1 is copied into one of two device slots while layer l computes."""

    def __init__(self, handle: Handle, slot_bytes: int):
        self._lib = handle._lib
        self._handle = handle
        s = ctypes.c_void_p()
        st = self._lib.lq_stream_create(ctypes.byref(s), handle.raw, int(slot_bytes))
        if st != LQ_OK:
            raise LQError(st, "lq_stream_create")
        self._s = s

    @staticmethod
    def problem(meta: dict, fmt: int, x, y) -> lq_problem:
        """One matrix of a layer: weight fields are byte offsets from pack_layer's `meta`."""
        p = lq_problem()
        p.format, p.M, p.N, p.K = fmt, int(x.shape[-2]), meta["N"], meta["K"]
        p.codes, p.scales, p.offsets = meta["codes"], meta["scales"], meta["offsets"]
        p.anchor_idx, p.anchor_w = meta["anchor_idx"], meta["anchor_w"]
        p.A, p.ld_anchor = meta["A"], meta["ld_anchor"]
        p.x, p.x_dtype, p.y, p.y_dtype = _ptr(x), _dtype_code(x), _ptr(y), _dtype_code(y)
        p.batch = 1
        return p

    def run(self, host_layers, host_stride: int, layer_bytes: int, L: int, problems, y_layer_stride: int = 0,
            stream=None):
        """host_layers: a uint8 CPU tensor (pinned for overlap) holding L layers at host_stride bytes."""
        arr = (lq_problem * len(problems))(*problems)
        st = self._lib.lq_stream_run(self._s, int(host_layers.data_ptr()), int(host_stride), int(layer_bytes), int(L),
                                     arr, len(problems), int(y_layer_stride), _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_stream_run")

    def run_direct(self, host_layers, host_stride: int, layer_bytes: int, L: int, problems, y_layer_stride: int = 0,
                   stream=None):
        """The same pass with the kernels reading the pinned host bytes directly (no copies)."""
        arr = (lq_problem * len(problems))(*problems)
        st = self._lib.lq_stream_run_direct(self._handle.raw, int(host_layers.data_ptr()), int(host_stride),
                                            int(layer_bytes), int(L), arr, len(problems), int(y_layer_stride),
                                            _stream(stream))
        if st != LQ_OK:
            raise LQError(st, "lq_stream_run_direct")

    def close(self):
        if getattr(self, "_s", None):
            st = self._lib.lq_stream_destroy(self._s)
            self._s = None
            if st != LQ_OK:
                raise LQError(st, "lq_stream_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
