"""Python binding of libkq, the quantized weight-streaming GEMV library for
GB300 (sm_103a).

Argument marshalling only: every function here checks nothing the C library
does not check itself, turns torch tensors (device memory, owned by the
caller) and streams into pointers, calls the entry point of the same name in
libkq.so and raises KQError on a non-zero status.  All arithmetic runs in the
library's CUDA kernels (or, for the offline host quantizers, in its C++ host
code); there is no fallback of any kind.

If the shared library has not been built, importing this package fails with
an ImportError: build it with ``quantized_weight_streaming_gb300.build.build()``
(or ``__graft_entry__.build()``).
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libkq.so is not built ({LIB_PATH} missing); run quantized_weight_streaming_gb300.build.build()")

_lib = ctypes.CDLL(LIB_PATH)

KQ_OK = 0
KQ_ERR_INVALID_ARG = 1
KQ_ERR_SHAPE = 2
KQ_ERR_ALIGNMENT = 3
KQ_ERR_NONFINITE = 4
KQ_ERR_RANGE = 5
KQ_ERR_WORKSPACE = 6
KQ_ERR_CUDA = 7
KQ_ERR_TIMEOUT = 8
KQ_ERR_UNSUPPORTED = 9

KQ_Q8_0 = 0
KQ_PQ2_0 = 1
KQ_PTQ1_0 = 2  # storage format: kq_prepare transcodes it to PQ2_0 planes
KQ_SCALE4 = 3  # scale4_gs32
FORMATS = {"q8_0": KQ_Q8_0, "pq2_0": KQ_PQ2_0, "ptq1_0": KQ_PTQ1_0, "scale4": KQ_SCALE4}


class KQError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _lib.kq_last_error().decode()
        super().__init__(f"{where}: {_lib.kq_status_string(status).decode()} ({status}): {msg}")


class kq_qmat(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("had_block", ctypes.c_int32), ("n", ctypes.c_int64),
                ("k", ctypes.c_int64), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("signs", ctypes.c_void_p)]


KQ_SRC_PACKED = 0
KQ_SRC_INPUT_OF = 1
KQ_SRC_OUTPUT_OF = 2


class kq_link(ctypes.Structure):
    _fields_ = [("src", ctypes.c_int32), ("stage", ctypes.c_int32), ("of", ctypes.c_int64),
                ("alpha", ctypes.c_float), ("reserved", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_QP = ctypes.POINTER(kq_qmat)

# name -> (restype, argtypes); every symbol declared in include/kq.h
SIGNATURES = {
    "kq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kq_last_error": (ctypes.c_char_p, []),
    "kq_version": (ctypes.c_int, []),
    "kq_block_size": (_I64, [ctypes.c_int]),
    "kq_blocks_bytes": (_I64, [ctypes.c_int, _I64, _I64]),
    "kq_scale_stride": (_I64, [ctypes.c_int, _I64]),
    "kq_codes_bytes": (_I64, [ctypes.c_int, _I64, _I64]),
    "kq_scales_bytes": (_I64, [ctypes.c_int, _I64, _I64]),
    "kq_quantize_q8_0": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "kq_quantize_pq2_0": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "kq_quantize_ptq1_0": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "kq_quantize_scale4": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "kq_quantize_scale4_device": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "kq_gemv_scale4": (ctypes.c_int, [_QP, _P, _P, _P, _SZ, _P]),
    "kq_gemv_f16": (ctypes.c_int, [_QP, _P, _P, _P, _SZ, _P]),
    "kq_hadamard_blockwise_host": (ctypes.c_int, [_P, _P, _I64, _I64, _I32]),
    "kq_prepare": (ctypes.c_int, [ctypes.c_int, _P, _I64, _I64, _P, _P, _P]),
    "kq_quantize_q8_0_device": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "kq_quantize_pq2_0_device": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "kq_dequantize": (ctypes.c_int, [_QP, _P, _P]),
    "kq_embed": (ctypes.c_int, [_QP, _P, _I64, _P, _P]),
    "kq_hadamard_blockwise": (ctypes.c_int, [_P, _P, _I64, _I64, _I32, _P]),
    "kq_rotate_blockwise_host": (ctypes.c_int, [_P, _P, _I64, _I64, _I32, _P]),
    "kq_rotate_blockwise": (ctypes.c_int, [_P, _P, _I64, _I64, _I32, _P, _P]),
    "kq_gemv_workspace_bytes": (_SZ, [_QP, _I64]),
    "kq_gemv_q8_0": (ctypes.c_int, [_QP, _P, _P, _P, _SZ, _P]),
    "kq_gemv_pq2_0": (ctypes.c_int, [_QP, _P, _P, _P, _SZ, _P]),
    "kq_gemm_small_m": (ctypes.c_int, [_QP, _P, _I64, _P, _P, _SZ, _P]),
    "kq_gemm_tc": (ctypes.c_int, [_QP, _P, _I64, _P, _I32, _P, _SZ, _P]),
    "kq_gemm_tc_workspace_bytes": (_SZ, [_QP, _I64, _I32]),
    "kq_gemm_splitk": (ctypes.c_int, [_QP, _P, _I64, _P, _I32, _P, _SZ, _P]),
    "kq_gemm_splitk_workspace_bytes": (_SZ, [_QP, _I64, _I32]),
    "kq_gemm_splitk_noalloc": (ctypes.c_int, [_QP, _P, _I64, _P, _I32, _P]),
    "kq_gemm_splitk_noalloc_max_bytes": (_SZ, []),
    "kq_decode_plan_create": (ctypes.c_int, [_QP, _I64, ctypes.POINTER(_P)]),
    "kq_decode_plan_create_linked": (ctypes.c_int, [_QP, ctypes.POINTER(kq_link), _I64, ctypes.POINTER(_P)]),
    "kq_decode_plan_stages": (ctypes.c_int, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "kq_decode_plan_sizes": (ctypes.c_int, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "kq_decode_workspace_bytes": (_SZ, [_P]),
    "kq_decode_step": (ctypes.c_int, [_P, _P, _P, _P, _SZ, _P]),
    "kq_decode_step_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _SZ, _P]),
    "kq_decode_plan_destroy": (None, [_P]),
    "kq_stream_read": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P]),
    "kq_selftest_bounded_wait": (ctypes.c_int, [_I64, _P]),
    "kq_device_status": (ctypes.c_int, [ctypes.c_int]),
    "kq_set_pq2_0_consumer": (ctypes.c_int, [ctypes.c_int]),
    "kq_get_pq2_0_consumer": (ctypes.c_int, []),
    "kq_kernel_binary_version": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
}

for _name, (_res, _args) in SIGNATURES.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def lib():
    return _lib


def _check(status, where):
    if status != KQ_OK:
        raise KQError(status, where)


def _ptr(t):
    """Address of a torch tensor, a numpy array or an integer (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _fmt(fmt):
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


# ---- layout ------------------------------------------------------------------

def kq_block_size(fmt):
    return _lib.kq_block_size(_fmt(fmt))


def kq_blocks_bytes(fmt, n, k):
    return _lib.kq_blocks_bytes(_fmt(fmt), n, k)


def kq_scale_stride(fmt, k):
    return _lib.kq_scale_stride(_fmt(fmt), k)


def kq_codes_bytes(fmt, n, k):
    return _lib.kq_codes_bytes(_fmt(fmt), n, k)


def kq_scales_bytes(fmt, n, k):
    return _lib.kq_scales_bytes(_fmt(fmt), n, k)


# ---- host quantizers (numpy in, numpy out) --------------------------------------

def kq_quantize_q8_0(w):
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    out = np.zeros(max(kq_blocks_bytes("q8_0", n, k), 1), dtype=np.uint8)
    _check(_lib.kq_quantize_q8_0(w.ctypes.data, n, k, out.ctypes.data), "kq_quantize_q8_0")
    return out[: n * (k // 32) * 34].reshape(n, k // 32, 34)


def kq_quantize_pq2_0(w_rot):
    w = np.ascontiguousarray(w_rot, dtype=np.float32)
    n, k = w.shape
    out = np.zeros(max(kq_blocks_bytes("pq2_0", n, k), 1), dtype=np.uint8)
    _check(_lib.kq_quantize_pq2_0(w.ctypes.data, n, k, out.ctypes.data), "kq_quantize_pq2_0")
    return out[: n * (k // 128) * 34].reshape(n, k // 128, 34)


def kq_quantize_scale4(w):
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    out = np.zeros(max(kq_blocks_bytes("scale4", n, k), 1), dtype=np.uint8)
    _check(_lib.kq_quantize_scale4(w.ctypes.data, n, k, out.ctypes.data), "kq_quantize_scale4")
    return out[: n * (k // 32) * 18].reshape(n, k // 32, 18)


def kq_quantize_ptq1_0(w_rot):
    w = np.ascontiguousarray(w_rot, dtype=np.float32)
    n, k = w.shape
    out = np.zeros(max(kq_blocks_bytes("ptq1_0", n, k), 1), dtype=np.uint8)
    _check(_lib.kq_quantize_ptq1_0(w.ctypes.data, n, k, out.ctypes.data), "kq_quantize_ptq1_0")
    return out[: n * (k // 128) * 28].reshape(n, k // 128, 28)


def kq_hadamard_blockwise_host(x, block=128):
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    out = np.empty_like(x2)
    _check(_lib.kq_hadamard_blockwise_host(x2.ctypes.data, out.ctypes.data, x2.shape[0], x2.shape[1], block),
           "kq_hadamard_blockwise_host")
    return out.reshape(x.shape)


# ---- device entry points (torch tensors) ------------------------------------------

class QMatrix:
    """A quantized matrix in device memory: torch tensors for the codes and
    scales planes plus the kq_qmat descriptor that points at them.  PQ2_0
    takes the rotation block (128, or the page's 1024) and an optional int8
    device tensor of k signs (kept referenced here)."""

    def __init__(self, fmt, n, k, device="cuda", had_block=None, signs=None):
        import torch

        self.fmt = _fmt(fmt)
        self.n, self.k = int(n), int(k)
        cb = kq_codes_bytes(self.fmt, n, k)
        sb = kq_scales_bytes(self.fmt, n, k)
        if cb <= 0 or sb <= 0:
            raise KQError(KQ_ERR_SHAPE, f"QMatrix({fmt}, {n}, {k})")
        self.codes = torch.empty(cb, dtype=torch.uint8, device=device)
        self.scales = torch.empty(sb // 2, dtype=torch.int16, device=device)
        if had_block is None:
            had_block = 128 if self.fmt == KQ_PQ2_0 else 0
        self.had_block = int(had_block)
        self.signs = signs
        self.desc = kq_qmat(self.fmt, self.had_block, self.n, self.k, self.codes.data_ptr(),
                            self.scales.data_ptr(), None if signs is None else signs.data_ptr())

    @property
    def nbytes(self):
        return self.codes.numel() + self.scales.numel() * 2

    @property
    def weight_bytes(self):
        """Bytes of the format itself (codes plus one fp16 scale per block)."""
        return self.codes.numel() + self.n * (self.k // kq_block_size(self.fmt)) * 2


def kq_prepare(W, d_blocks, stream=None, block_fmt=None):
    """Blocks (device memory) -> W's planes; block_fmt="ptq1_0" transcodes
    PTQ1_0 blocks into a PQ2_0 matrix."""
    fmt = W.fmt if block_fmt is None else _fmt(block_fmt)
    _check(_lib.kq_prepare(fmt, _ptr(d_blocks), W.n, W.k, W.codes.data_ptr(), W.scales.data_ptr(), _stream(stream)),
           "kq_prepare")


def kq_quantize_q8_0_device(W, d_w, stream=None):
    _check(_lib.kq_quantize_q8_0_device(_ptr(d_w), W.n, W.k, W.codes.data_ptr(), W.scales.data_ptr(),
                                        _stream(stream)), "kq_quantize_q8_0_device")


def kq_quantize_pq2_0_device(W, d_w_rot, stream=None):
    _check(_lib.kq_quantize_pq2_0_device(_ptr(d_w_rot), W.n, W.k, W.codes.data_ptr(), W.scales.data_ptr(),
                                         _stream(stream)), "kq_quantize_pq2_0_device")


def kq_quantize_scale4_device(W, d_w, stream=None):
    _check(_lib.kq_quantize_scale4_device(_ptr(d_w), W.n, W.k, W.codes.data_ptr(), W.scales.data_ptr(),
                                          _stream(stream)), "kq_quantize_scale4_device")


def kq_embed(E, d_ids, count, d_out, stream=None):
    """Rows d_ids of the quantized table E, dequantized (and inverse-rotated for PQ2_0)."""
    _check(_lib.kq_embed(ctypes.byref(E.desc), _ptr(d_ids), count, _ptr(d_out), _stream(stream)), "kq_embed")


def kq_dequantize(W, d_out, stream=None):
    _check(_lib.kq_dequantize(ctypes.byref(W.desc), _ptr(d_out), _stream(stream)), "kq_dequantize")


def kq_hadamard_blockwise(d_in, d_out, rows, k, block=128, stream=None):
    _check(_lib.kq_hadamard_blockwise(_ptr(d_in), _ptr(d_out), rows, k, block, _stream(stream)),
           "kq_hadamard_blockwise")


def kq_rotate_blockwise(d_in, d_out, rows, k, block, d_signs=None, stream=None):
    _check(_lib.kq_rotate_blockwise(_ptr(d_in), _ptr(d_out), rows, k, block, _ptr(d_signs), _stream(stream)),
           "kq_rotate_blockwise")


def kq_rotate_blockwise_host(x, block, signs=None):
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    out = np.empty_like(x2)
    sg = None if signs is None else np.ascontiguousarray(signs, dtype=np.int8)
    _check(_lib.kq_rotate_blockwise_host(x2.ctypes.data, out.ctypes.data, x2.shape[0], x2.shape[1], block,
                                         None if sg is None else sg.ctypes.data), "kq_rotate_blockwise_host")
    return out.reshape(x.shape)


def kq_gemv_workspace_bytes(W, m=1):
    return _lib.kq_gemv_workspace_bytes(ctypes.byref(W.desc), m)


def kq_gemm_splitk_workspace_bytes(W, m, splits):
    return _lib.kq_gemm_splitk_workspace_bytes(ctypes.byref(W.desc), m, splits)


def _ws(ws):
    if ws is None:
        return None, 0
    return _ptr(ws), ws.numel() * ws.element_size()


def kq_gemv_q8_0(W, d_x, d_y, ws=None, stream=None):
    p, nb = _ws(ws)
    _check(_lib.kq_gemv_q8_0(ctypes.byref(W.desc), _ptr(d_x), _ptr(d_y), p, nb, _stream(stream)), "kq_gemv_q8_0")


def kq_gemv_scale4(W, d_x, d_y, ws=None, stream=None):
    p, nb = _ws(ws)
    _check(_lib.kq_gemv_scale4(ctypes.byref(W.desc), _ptr(d_x), _ptr(d_y), p, nb, _stream(stream)), "kq_gemv_scale4")


def kq_gemv_f16(W, d_x16, d_y16, ws=None, stream=None):
    """The fp16 chain: fp16 activation in, fp16 output (any format)."""
    p, nb = _ws(ws)
    _check(_lib.kq_gemv_f16(ctypes.byref(W.desc), _ptr(d_x16), _ptr(d_y16), p, nb, _stream(stream)), "kq_gemv_f16")


def kq_gemv_pq2_0(W, d_x, d_y, ws=None, stream=None):
    p, nb = _ws(ws)
    _check(_lib.kq_gemv_pq2_0(ctypes.byref(W.desc), _ptr(d_x), _ptr(d_y), p, nb, _stream(stream)), "kq_gemv_pq2_0")


def kq_gemm_small_m(W, d_X, m, d_Y, ws=None, stream=None):
    p, nb = _ws(ws)
    _check(_lib.kq_gemm_small_m(ctypes.byref(W.desc), _ptr(d_X), m, _ptr(d_Y), p, nb, _stream(stream)),
           "kq_gemm_small_m")


def kq_gemm_tc_workspace_bytes(W, m, splits=0):
    return _lib.kq_gemm_tc_workspace_bytes(ctypes.byref(W.desc), m, splits)


def kq_gemm_tc(W, d_X, m, d_Y, splits=0, ws=None, stream=None):
    """Small-batch GEMM on the tensor cores (tcgen05)."""
    p, nb = _ws(ws)
    _check(_lib.kq_gemm_tc(ctypes.byref(W.desc), _ptr(d_X), m, _ptr(d_Y), splits, p, nb, _stream(stream)),
           "kq_gemm_tc")


def kq_gemm_splitk(W, d_X, m, d_Y, splits, ws=None, stream=None):
    p, nb = _ws(ws)
    _check(_lib.kq_gemm_splitk(ctypes.byref(W.desc), _ptr(d_X), m, _ptr(d_Y), splits, p, nb, _stream(stream)),
           "kq_gemm_splitk")


def kq_kernel_binary_version():
    v = ctypes.c_int()
    _check(_lib.kq_kernel_binary_version(ctypes.byref(v)), "kq_kernel_binary_version")
    return v.value


def kq_gemm_splitk_noalloc(W, d_X, m, d_Y, splits, stream=None):
    """Split-K GEMM whose partial sums use the library's static device scratch
    (no workspace argument, no allocation)."""
    _check(_lib.kq_gemm_splitk_noalloc(ctypes.byref(W.desc), _ptr(d_X), m, _ptr(d_Y), splits, _stream(stream)),
           "kq_gemm_splitk_noalloc")


def kq_gemm_splitk_noalloc_max_bytes():
    return _lib.kq_gemm_splitk_noalloc_max_bytes()


def kq_selftest_bounded_wait(limit_cycles, stream=None):
    _check(_lib.kq_selftest_bounded_wait(int(limit_cycles), _stream(stream)), "kq_selftest_bounded_wait")


def kq_stream_read(d_src, nbytes, d_sink, stage_bytes=34816, stages=4, stream=None):
    """Read-only streaming control: stream nbytes of d_src once through shared
    memory; XORs the XOR of its 32-bit words into d_sink[0]."""
    _check(_lib.kq_stream_read(_ptr(d_src), nbytes, stage_bytes, stages, _ptr(d_sink), _stream(stream)),
           "kq_stream_read")


def kq_device_status(clear=True):
    return _lib.kq_device_status(1 if clear else 0)


KQ_PQ2_0_MMA_SYNC = 0
KQ_PQ2_0_TCGEN05 = 1


def kq_set_pq2_0_consumer(consumer):
    """Selects the consumer of PQ2_0 products at one activation row
    (KQ_PQ2_0_MMA_SYNC, the default, or KQ_PQ2_0_TCGEN05); process-wide."""
    _check(_lib.kq_set_pq2_0_consumer(int(consumer)), "kq_set_pq2_0_consumer")


def kq_get_pq2_0_consumer():
    return _lib.kq_get_pq2_0_consumer()


class DecodePlan:
    """kq_decode_plan_create (or, with links, kq_decode_plan_create_linked) /
    kq_decode_step / kq_decode_plan_destroy.  links: one (src, stage, of,
    alpha) tuple per matrix."""

    def __init__(self, mats, links=None):
        self.mats = list(mats)
        arr = (kq_qmat * len(self.mats))(*[m.desc for m in self.mats])
        h = ctypes.c_void_p()
        if links is None:
            _check(_lib.kq_decode_plan_create(arr, len(self.mats), ctypes.byref(h)), "kq_decode_plan_create")
        else:
            links = list(links)
            la = (kq_link * len(links))(*[kq_link(int(src), int(stage), int(of), float(alpha), 0)
                                          for src, stage, of, alpha in links])
            _check(_lib.kq_decode_plan_create_linked(arr, la, len(links), ctypes.byref(h)),
                   "kq_decode_plan_create_linked")
        self.handle = h
        st, ns = _I32(), _I32()
        _check(_lib.kq_decode_plan_stages(h, ctypes.byref(st), ctypes.byref(ns)), "kq_decode_plan_stages")
        self.stages, self.split_matrices = st.value, ns.value
        xf, yf, wb = _I64(), _I64(), _I64()
        _check(_lib.kq_decode_plan_sizes(h, ctypes.byref(xf), ctypes.byref(yf), ctypes.byref(wb)),
               "kq_decode_plan_sizes")
        self.x_floats, self.y_floats, self.weight_bytes = xf.value, yf.value, wb.value
        self.workspace_bytes = _lib.kq_decode_workspace_bytes(h)

    def step(self, d_x_packed, d_y_packed, ws=None, stream=None):
        p, nb = _ws(ws)
        _check(_lib.kq_decode_step(self.handle, _ptr(d_x_packed), _ptr(d_y_packed), p, nb, _stream(stream)),
               "kq_decode_step")

    def step_host(self, h_x_packed, h_y_packed, d_x_packed, d_y_packed, ws=None, stream=None):
        """kq_decode_step_host: host (ideally pinned) CPU tensors in and out,
        through the given device buffers; asynchronous on `stream`.  A pinned
        h_x_packed is read by the kernel in place (d_x_packed is then left
        unwritten), and a one-stage plan writes a pinned h_y_packed directly
        (d_y_packed is then left unwritten)."""
        p, nb = _ws(ws)
        _check(_lib.kq_decode_step_host(self.handle, _ptr(h_x_packed), _ptr(h_y_packed), _ptr(d_x_packed),
                                        _ptr(d_y_packed), p, nb, _stream(stream)), "kq_decode_step_host")

    def close(self):
        if self.handle:
            _lib.kq_decode_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
