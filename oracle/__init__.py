"""FP64 CPU oracle of the quantized weight-streaming GEMV (ctypes wrapper of
oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline may import this package; the product library never does, and the
product path must fail loudly rather than fall back to it.

Definitions followed (details and citations in oracle.h):

* Q8_0 -- "Kipp Architecture", section "Weight quantization": 32-weight blocks,
  fp16 scale d and int8 codes, value d*q, quantized against the fp16-rounded
  scale.
* PQ2_0 -- "Bonsai 2 27B - ternary g128 + blockwise Hadamard", section 3.1:
  128-weight 34-byte blocks, 2-bit codes at bit offset 2*(j%4), value
  (q-1)*d, d = max|w|, q = round(w/d) + 1.
* Rotation -- same page, sections 4.1-4.2: R = H_n / sqrt(n) (Sylvester,
  natural order) block-diagonal along K; W' = W R^T is stored (rotate, then
  quantize); the activation gets x' = R x before the product.

Outputs of the GEMV are FP64 sums with the per-row acceptance scale
absdot_i = sum_j |w_ij x_j|; a result passes when |y - y_oracle| <= 1e-4 *
absdot_i.
"""
import ctypes
import os

import numpy as np

from . import build as _build

ORC_OK, ORC_ERR_SHAPE, ORC_ERR_NONFINITE, ORC_ERR_RANGE = 0, 1, 2, 3
Q8_0_QK, PQ2_0_QK, BLOCK_BYTES = 32, 128, 34
HADAMARD_N = 128
TOLERANCE = 1e-4

_lib = None


class OracleError(RuntimeError):
    pass


def lib():
    global _lib
    if _lib is None:
        _build.build()
        L = ctypes.CDLL(_build.LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.orc_half_from_float.argtypes = [ctypes.c_float]
        L.orc_half_from_float.restype = ctypes.c_uint16
        L.orc_float_from_half.argtypes = [ctypes.c_uint16]
        L.orc_float_from_half.restype = ctypes.c_float
        L.orc_half_from_float_array.argtypes = [P, I64, P]
        L.orc_float_from_half_array.argtypes = [P, I64, P]
        for name in ("orc_q8_0_quantize", "orc_q8_0_dequant", "orc_pq2_0_quantize", "orc_pq2_0_dequant"):
            getattr(L, name).argtypes = [P, I64, I64, P]
            getattr(L, name).restype = ctypes.c_int
        for name in ("orc_ptq1_0_quantize", "orc_ptq1_0_dequant", "orc_scale4_quantize", "orc_scale4_dequant"):
            getattr(L, name).argtypes = [P, I64, I64, P]
            getattr(L, name).restype = ctypes.c_int
        L.orc_ptq1_0_encode_byte.argtypes = [P]
        L.orc_ptq1_0_encode_byte.restype = ctypes.c_int
        L.orc_ptq1_0_decode_trit.argtypes = [ctypes.c_int32, ctypes.c_int32]
        L.orc_ptq1_0_decode_trit.restype = ctypes.c_int
        L.orc_hadamard.argtypes = [ctypes.c_int32, P]
        L.orc_hadamard.restype = ctypes.c_int
        L.orc_rotate_rows.argtypes = [P, I64, I64, ctypes.c_int32, P, P]
        L.orc_rotate_rows.restype = ctypes.c_int
        L.orc_rotate_rows_signed.argtypes = [P, I64, I64, ctypes.c_int32, P, P, P]
        L.orc_rotate_rows_signed.restype = ctypes.c_int
        L.orc_rotate_rows_inverse.argtypes = [P, I64, I64, ctypes.c_int32, P, P]
        L.orc_rotate_rows_inverse.restype = ctypes.c_int
        L.orc_gemv_f64.argtypes = [P, I64, I64, P, P, I64, ctypes.c_int32, P, P]
        L.orc_gemv_f64.restype = ctypes.c_int
        L.orc_max_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_set_threads.restype = None
        _lib = L
    return _lib


def _check(rc, what):
    if rc != ORC_OK:
        raise OracleError(f"{what}: oracle status {rc}")


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def max_threads():
    return lib().orc_max_threads()


def set_threads(n):
    """Threads of the row loops from now on (timing only; results do not
    depend on it)."""
    lib().orc_set_threads(int(n))


# -- binary16 -----------------------------------------------------------------

def half_bits(values):
    v = _f32(values).ravel()
    out = np.empty(v.size, dtype=np.uint16)
    lib().orc_half_from_float_array(v.ctypes.data, v.size, out.ctypes.data)
    return out.reshape(np.shape(values))


def half_value(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(b.size, dtype=np.float32)
    lib().orc_float_from_half_array(b.ctypes.data, b.size, out.ctypes.data)
    return out.reshape(np.shape(bits))


# -- formats ------------------------------------------------------------------

def q8_0_quantize(w):
    """n x k fp32 -> uint8 array [n, k/32, 34] of Q8_0 blocks."""
    w = _f32(w)
    n, k = w.shape
    if k % Q8_0_QK:
        raise OracleError("k % 32 != 0")
    out = np.zeros((n, k // Q8_0_QK, BLOCK_BYTES), dtype=np.uint8)
    _check(lib().orc_q8_0_quantize(w.ctypes.data, n, k, out.ctypes.data), "q8_0_quantize")
    return out


def q8_0_dequant(blocks, n, k):
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty((n, k), dtype=np.float32)
    _check(lib().orc_q8_0_dequant(b.ctypes.data, n, k, out.ctypes.data), "q8_0_dequant")
    return out


def pq2_0_quantize(w_rot):
    """Rotated n x k fp32 -> uint8 array [n, k/128, 34] of PQ2_0 blocks."""
    w = _f32(w_rot)
    n, k = w.shape
    if k % PQ2_0_QK:
        raise OracleError("k % 128 != 0")
    out = np.zeros((n, k // PQ2_0_QK, BLOCK_BYTES), dtype=np.uint8)
    _check(lib().orc_pq2_0_quantize(w.ctypes.data, n, k, out.ctypes.data), "pq2_0_quantize")
    return out


def pq2_0_dequant(blocks, n, k):
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty((n, k), dtype=np.float32)
    _check(lib().orc_pq2_0_dequant(b.ctypes.data, n, k, out.ctypes.data), "pq2_0_dequant")
    return out


def ptq1_0_quantize(w_rot):
    """PTQ1_0 blocks [n, k/128, 28] of already rotated weights."""
    w = _f32(w_rot)
    n, k = w.shape
    out = np.zeros((n, k // 128, 28), dtype=np.uint8)
    _check(lib().orc_ptq1_0_quantize(w.ctypes.data, n, k, out.ctypes.data), "ptq1_0_quantize")
    return out


def ptq1_0_dequant(blocks, n, k):
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty((n, k), dtype=np.float32)
    _check(lib().orc_ptq1_0_dequant(b.ctypes.data, n, k, out.ctypes.data), "ptq1_0_dequant")
    return out


def scale4_quantize(w):
    """scale4_gs32 blocks [n, k/32, 18]."""
    w = _f32(w)
    n, k = w.shape
    out = np.zeros((n, k // 32, 18), dtype=np.uint8)
    _check(lib().orc_scale4_quantize(w.ctypes.data, n, k, out.ctypes.data), "scale4_quantize")
    return out


def scale4_dequant(blocks, n, k):
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty((n, k), dtype=np.float32)
    _check(lib().orc_scale4_dequant(b.ctypes.data, n, k, out.ctypes.data), "scale4_dequant")
    return out


def scale4_reference(w, x):
    """Quantize W to scale4_gs32 and return (blocks, dequantized W, y, absdot)."""
    w = _f32(w)
    n, k = w.shape
    blocks = scale4_quantize(w)
    deq = scale4_dequant(blocks, n, k)
    x = np.asarray(x, dtype=np.float32)
    if x.ndim == 1:
        y, a = gemv(deq, x.astype(np.float64))
    else:
        y, a = gemm(deq, x.astype(np.float64))
    return blocks, deq, y, a


def ptq1_0_encode_byte(trits):
    t = np.ascontiguousarray(trits, dtype=np.int32)
    return lib().orc_ptq1_0_encode_byte(t.ctypes.data)


def ptq1_0_decode_trit(q, n):
    return lib().orc_ptq1_0_decode_trit(int(q), int(n))


# -- rotation -----------------------------------------------------------------

def hadamard(n):
    """Unnormalised Sylvester Hadamard matrix H_n (entries +-1), FP64."""
    out = np.empty((n, n), dtype=np.float64)
    _check(lib().orc_hadamard(int(n), out.ctypes.data), "hadamard")
    return out


def rotate_rows(x, n=HADAMARD_N, signs=None):
    """Blockwise R = H_n S / sqrt(n) along the last axis (S = diag(signs), the
    identity when signs is None).  Returns (fp64, fp32)."""
    x = _f32(x)
    shape = x.shape
    x2 = x.reshape(-1, shape[-1])
    rows, k = x2.shape
    o64 = np.empty((rows, k), dtype=np.float64)
    o32 = np.empty((rows, k), dtype=np.float32)
    if signs is None:
        sp = None
    else:
        sg = np.ascontiguousarray(signs, dtype=np.int8)
        if sg.shape != (k,):
            raise OracleError("signs length mismatch")
        sp = sg.ctypes.data
    _check(lib().orc_rotate_rows_signed(x2.ctypes.data, rows, k, int(n), sp, o64.ctypes.data, o32.ctypes.data),
           "rotate_rows")
    return o64.reshape(shape), o32.reshape(shape)


def rotate_rows_inverse(z, n=HADAMARD_N, signs=None):
    """e = R^T z = S (H_n z) / sqrt(n) per n-block along the last axis (FP64)."""
    z = _f32(z)
    shape = z.shape
    z2 = z.reshape(-1, shape[-1])
    rows, k = z2.shape
    out = np.empty((rows, k), dtype=np.float64)
    sp = None
    if signs is not None:
        sg = np.ascontiguousarray(signs, dtype=np.int8)
        if sg.shape != (k,):
            raise OracleError("signs length mismatch")
        sp = sg.ctypes.data
    _check(lib().orc_rotate_rows_inverse(z2.ctypes.data, rows, k, int(n), sp, out.ctypes.data), "rotate_rows_inverse")
    return out.reshape(shape)


def embed_reference(fmt, blocks, vocab, dim, ids, had=HADAMARD_N, signs=None):
    """Rows `ids` of a quantized table (blocks of the stored rows), dequantized;
    for PQ2_0 the stored rows are R e, so e = R^T z (transform, then signs).
    Returns (FP64 rows, per-row-block sum |z| for the error bound)."""
    deq = {"q8_0": q8_0_dequant, "pq2_0": pq2_0_dequant, "scale4": scale4_dequant}[fmt](blocks, vocab, dim)
    z = deq[np.asarray(ids)]
    if fmt != "pq2_0":
        return z.astype(np.float64), None
    e = rotate_rows_inverse(z, had, signs)
    blk = np.abs(z.astype(np.float64)).reshape(len(ids), -1, had).sum(axis=2).repeat(had, axis=1)
    return e, blk


# -- GEMV ---------------------------------------------------------------------

def gemv(w, x64, rows=None, rows_are_packed=False, n_total=None):
    """FP64 y = W x and absdot = |W| |x| (elementwise products) for the listed
    rows of W (all rows when rows is None)."""
    w = _f32(w)
    x = np.ascontiguousarray(x64, dtype=np.float64)
    k = w.shape[1]
    if x.shape != (k,):
        raise OracleError("x length mismatch")
    if rows is None:
        n = w.shape[0]
        r_ptr, nr = None, n
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n = n_total if n_total is not None else w.shape[0]
        r_ptr, nr = r.ctypes.data, r.size
    y = np.empty(nr, dtype=np.float64)
    a = np.empty(nr, dtype=np.float64)
    _check(lib().orc_gemv_f64(w.ctypes.data, n, k, x.ctypes.data, r_ptr, nr, int(bool(rows_are_packed)),
                              y.ctypes.data, a.ctypes.data), "gemv")
    return y, a


def gemm(w, X64):
    """Y[m] = W x_m for each activation row (FP64), with the matching absdot."""
    X = np.atleast_2d(np.asarray(X64, dtype=np.float64))
    ys, As = [], []
    for m in range(X.shape[0]):
        y, a = gemv(w, X[m])
        ys.append(y)
        As.append(a)
    return np.stack(ys), np.stack(As)


# -- whole pipelines from unquantized weights -----------------------------------

def q8_0_reference(w, x):
    """Quantize W (fp32 n x k) to Q8_0 and return (blocks, dequantized W,
    y, absdot) for activation x (or rows of X)."""
    w = _f32(w)
    n, k = w.shape
    blocks = q8_0_quantize(w)
    deq = q8_0_dequant(blocks, n, k)
    x = np.asarray(x, dtype=np.float32)
    if x.ndim == 1:
        y, a = gemv(deq, x.astype(np.float64))
    else:
        y, a = gemm(deq, x.astype(np.float64))
    return blocks, deq, y, a


def pq2_0_reference(w, x):
    """Rotate W blockwise (fp32), quantize to PQ2_0, rotate x in FP64 and
    return (blocks, dequantized W', y, absdot)."""
    w = _f32(w)
    n, k = w.shape
    _, w_rot = rotate_rows(w)
    blocks = pq2_0_quantize(w_rot)
    deq = pq2_0_dequant(blocks, n, k)
    x = np.asarray(x, dtype=np.float32)
    x_rot64, _ = rotate_rows(x)
    if x.ndim == 1:
        y, a = gemv(deq, x_rot64)
    else:
        y, a = gemm(deq, x_rot64)
    return blocks, deq, y, a


def reference(fmt, w, x):
    if fmt == "q8_0":
        return q8_0_reference(w, x)
    if fmt == "scale4":
        return scale4_reference(w, x)
    if fmt == "pq2_0":
        return pq2_0_reference(w, x)
    raise OracleError(fmt)


def f16_chain_reference(fmt, w, x16, had=HADAMARD_N, signs=None):
    """The fp16 activation chain of the Bonsai page, section 4.4: activation
    fp16 -> fp32 (sign flip and) transform -> fp16 -> product accumulated in
    fp32 -> fp16 output.  Reading: the transformed activation is the exact
    (FP64) R x rounded once to fp16; an fp32 transform may land on the other
    fp16 neighbour when R x lies within the fp32 transform's error bound
    ((log2 n + 3) 2^-24 sum_blk |x| / sqrt(n)) of a rounding midpoint, and
    `slack` bounds that: sum_j |w_ij| * (the fp16 step at x'_j) over those j.
    x16: fp16 values (numpy float16).  Returns (y FP64, absdot, slack, x'16)."""
    w = _f32(w)
    n, k = w.shape
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    if fmt == "pq2_0":
        _, w_rot = rotate_rows(w, had, signs)
        deq = pq2_0_dequant(pq2_0_quantize(w_rot), n, k)
        xr64, _ = rotate_rows(x, had, signs)
        xp16 = xr64.astype(np.float16)  # one rounding of the exact value (to nearest even)
        # where an fp32 transform could have rounded to the other neighbour
        blk_abs = np.abs(x.astype(np.float64)).reshape(-1, had).sum(axis=1).repeat(had)
        eps = (np.log2(had) + 3) * 2.0 ** -24 * blk_abs / np.sqrt(had)
        lo = np.nextafter(xp16, np.float16(-np.inf)).astype(np.float64)
        hi = np.nextafter(xp16, np.float16(np.inf)).astype(np.float64)
        c = xp16.astype(np.float64)
        near = np.minimum(np.abs(xr64 - (c + lo) / 2), np.abs(xr64 - (c + hi) / 2)) <= eps
        step = np.where(near, np.maximum(c - lo, hi - c), 0.0)
    else:
        deq = (q8_0_dequant(q8_0_quantize(w), n, k) if fmt == "q8_0" else scale4_dequant(scale4_quantize(w), n, k))
        xp16 = x.astype(np.float16)
        step = np.zeros(k)
    y, a = gemv(deq, xp16.astype(np.float64))
    slack = np.abs(deq.astype(np.float64)) @ step
    return y, a, slack, xp16


def within_bound(y, y_ref, absdot, tol=TOLERANCE):
    """Per-row acceptance: |y - y_ref| <= tol * absdot.  Returns (ok, worst
    ratio of error to bound)."""
    err = np.abs(np.asarray(y, dtype=np.float64) - y_ref)
    bound = tol * np.asarray(absdot, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0.0))
    return bool(np.all(err <= bound)), float(ratio.max()) if ratio.size else 0.0
