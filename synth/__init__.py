"""Seeded synthetic inputs for the quantized weight-streaming GEMV.

This module holds no arithmetic of the method.  It turns (seed, stream,
element index) into fp32 values with a counter-based generator (Philox4x64-10
with an Irwin-Hall sum of twelve uniforms, see philox.h), identical on the host
(``fill_host``) and on the device (``fill_device``), and it describes the
workload shapes:

* ``q8_0_gemv``     Q8_0 GEMV, W 1024 x 2560, x 2560
* ``pq2_0_gemv``    PQ2_0 GEMV with blockwise Hadamard, W 10240 x 5120, x 5120
* ``qwen3_4b_q8_0_step``      Qwen3-4B-shaped list of 253 Q8_0 projections
* ``bonsai_27b_pq2_0_step``   Bonsai-27B-shaped list of 401 PQ2_0 projections
* ``qwen3_4b_scale4_step``    the same 253 projections in scale4_gs32
* ``small_m``       M in {1, 4, 16, 64} activation rows against Q8_0 2560->9728
                    and PQ2_0 5120->17408

Weights are about N(0, 0.02) on a 2^-20 grid, activations about N(0, 1) on a
2^-16 grid.  The shapes stand in for the real checkpoints (Qwen3-4B and
Bonsai 2 27B), which are not used.
"""
import ctypes
import os

import numpy as np

from . import build as _build

W_RANGE, W_EXP2 = 20972, 20
X_RANGE, X_EXP2 = 65536, 16

ROLE_W = 0
ROLE_X = 1
ROLE_S = 2  # sign vectors of a rotation, indexed by K width

CONFIG_IDS = {
    "q8_0_gemv": 0,
    "pq2_0_gemv": 1,
    "qwen3_4b_q8_0_step": 2,
    "bonsai_27b_pq2_0_step": 3,
    "small_m": 4,
    "qwen3_4b_scale4_step": 5,
    "test": 7,
}

Q8_0 = "q8_0"
PQ2_0 = "pq2_0"
SCALE4 = "scale4"


def stream_id(config, role, index=0):
    """Stream number of one tensor of a workload: config, role (weights or
    activation) and the tensor's index within the workload."""
    cid = CONFIG_IDS[config] if isinstance(config, str) else int(config)
    return (cid << 40) | (int(role) << 32) | int(index)


# --------------------------------------------------------------------------
# Workload shapes.  A projection is (name, fmt, n_out, k_in).
# --------------------------------------------------------------------------

def qwen3_4b_projections():
    """Qwen3-4B-shaped decode step: 36 layers of q/k/v/o/gate/up/down, then
    the lm_head; 253 matrices, 4,022,272,000 weights."""
    mats = []
    for layer in range(36):
        for name, n, k in (("q_proj", 4096, 2560), ("k_proj", 1024, 2560), ("v_proj", 1024, 2560),
                           ("o_proj", 2560, 4096), ("gate_proj", 9728, 2560), ("up_proj", 9728, 2560),
                           ("down_proj", 2560, 9728)):
            mats.append((f"layers.{layer}.{name}", Q8_0, n, k))
    mats.append(("lm_head", Q8_0, 151936, 2560))
    return mats


def bonsai_27b_projections():
    """Bonsai-27B-shaped decode weight stream, in model order: 64 layers, of
    which layers 3, 7, ..., 63 are full attention (q 5120->12288, k and v
    5120->1024, o 6144->5120) and the other 48 are gated-delta-net layers
    (qkv 5120->10240, z 5120->6144, out 6144->5120); every layer ends with an
    FFN (gate and up 5120->17408, down 17408->5120); then the output head
    5120->248320.  401 matrices, 25,598,361,600 weights."""
    mats = []
    for layer in range(64):
        if layer % 4 == 3:
            parts = (("attn_q", 12288, 5120), ("attn_k", 1024, 5120), ("attn_v", 1024, 5120),
                     ("attn_output", 5120, 6144))
        else:
            parts = (("attn_qkv", 10240, 5120), ("attn_gate", 6144, 5120), ("ssm_out", 5120, 6144))
        for name, n, k in parts + (("ffn_gate", 17408, 5120), ("ffn_up", 17408, 5120), ("ffn_down", 5120, 17408)):
            mats.append((f"blk.{layer}.{name}", PQ2_0, n, k))
    mats.append(("output", PQ2_0, 248320, 5120))
    return mats


# --------------------------------------------------------------------------
# Dependency structure of a decode step (linked decode plans).  A link is
# (src, stage, of, alpha), src one of the kinds below (the values of the C
# ABI's kq_src_kind).  The non-projection operations between projections
# (attention, norms, activation functions, residuals) are outside the
# library; each dependent activation is alpha times an earlier projection's
# output, alpha = 1 / (sigma_w sqrt(k_src)) with sigma_w the spread of the
# quantized synthetic weights, so that activations stay near unit scale
# along the chain.
# --------------------------------------------------------------------------
SRC_PACKED = 0
SRC_INPUT_OF = 1
SRC_OUTPUT_OF = 2
W_STD_EFF = {Q8_0: 0.0200, PQ2_0: 0.0222, SCALE4: 0.0200}  # std of the dequantized N(0, 0.02) weights


def chain_alpha(fmt, k_src):
    """fp32 scale of the successor activation of a projection with input length k_src."""
    return float(np.float32(1.0 / (W_STD_EFF[fmt] * np.sqrt(k_src))))


def decode_links(config):
    """One link per projection of a decode-step workload, in list order: the
    layer's input feeds its first projection group (q/k/v, or GDN qkv/z),
    the attention output projection reads q's output (prefix) or z's, the FFN
    gate/up group reads the output projection, down reads up, the next layer
    reads down, and the head reads the last down.  Stage 4l..4l+3 per layer l."""
    mats = workload(config)
    names = [m[0] for m in mats]
    idx = {name: i for i, name in enumerate(names)}

    def out_of(j, stage):
        _, fmt, _, k = mats[j]
        return (SRC_OUTPUT_OF, stage, j, chain_alpha(fmt, k))

    links = [None] * len(mats)
    prev = None  # index of the previous layer's down projection
    if config in ("qwen3_4b_q8_0_step", "qwen3_4b_scale4_step"):
        layers, pre = 36, "layers."
        groups = lambda l: (("q_proj", "k_proj", "v_proj"), "q_proj", "o_proj", "gate_proj", "up_proj", "down_proj")
        head = "lm_head"
    elif config == "bonsai_27b_pq2_0_step":
        layers, pre = 64, "blk."

        def groups(l):
            if l % 4 == 3:
                return (("attn_q", "attn_k", "attn_v"), "attn_q", "attn_output", "ffn_gate", "ffn_up", "ffn_down")
            return (("attn_qkv", "attn_gate"), "attn_gate", "ssm_out", "ffn_gate", "ffn_up", "ffn_down")

        head = "output"
    else:
        raise KeyError(config)
    for l in range(layers):
        first, o_src, o_name, g_name, u_name, d_name = groups(l)
        at = lambda n: idx[f"{pre}{l}.{n}"]
        s0 = 4 * l
        root = at(first[0])
        links[root] = (SRC_PACKED, s0, 0, 1.0) if prev is None else out_of(prev, s0)
        for n in first[1:]:
            links[at(n)] = (SRC_INPUT_OF, s0, root, 1.0)
        links[at(o_name)] = out_of(at(o_src), s0 + 1)
        links[at(g_name)] = out_of(at(o_name), s0 + 2)
        links[at(u_name)] = (SRC_INPUT_OF, s0 + 2, at(g_name), 1.0)
        links[at(d_name)] = out_of(at(u_name), s0 + 3)
        prev = at(d_name)
    links[idx[head]] = out_of(prev, 4 * layers)
    assert all(lk is not None for lk in links)
    return links


SMALL_M_VALUES = (1, 4, 16, 64)
SMALL_M_MATRICES = (("q8_0_2560x9728", Q8_0, 9728, 2560), ("pq2_0_5120x17408", PQ2_0, 17408, 5120))


def workload(config):
    """List of projections (name, fmt, n, k) of a workload."""
    if config == "q8_0_gemv":
        return [("w", Q8_0, 1024, 2560)]
    if config == "pq2_0_gemv":
        return [("w", PQ2_0, 10240, 5120)]
    if config == "qwen3_4b_q8_0_step":
        return qwen3_4b_projections()
    if config == "bonsai_27b_pq2_0_step":
        return bonsai_27b_projections()
    if config == "small_m":
        return list(SMALL_M_MATRICES)
    if config == "qwen3_4b_scale4_step":  # the Qwen3-4B projections in scale4_gs32
        return [(name, SCALE4, n, k) for name, _, n, k in qwen3_4b_projections()]
    raise KeyError(config)


def small_m_x_index(mat_index, m):
    """Activation tensor index of the small-M workload for matrix mat_index and
    M rows."""
    return mat_index * 1000 + m


# --------------------------------------------------------------------------
# Generators
# --------------------------------------------------------------------------

_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        _build.build()
        lib = ctypes.CDLL(_build.HOST_LIB)
        lib.synth_fill_host.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32]
        lib.synth_fill_host.restype = None
        lib.synth_philox_block.argtypes = [ctypes.c_void_p] * 3
        lib.synth_philox_block.restype = None
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        _build.build()
        lib = ctypes.CDLL(_build.DEV_LIB)
        lib.synth_fill_device.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_void_p]
        lib.synth_fill_device.restype = ctypes.c_int
        _dev = lib
    return _dev


def _params(kind):
    if kind == "w":
        return W_RANGE, W_EXP2
    if kind == "x":
        return X_RANGE, X_EXP2
    raise ValueError(kind)


def philox_block(ctr, key):
    """Raw Philox4x64-10 block (4 uint64) for a counter (4 uint64) and key (2 uint64)."""
    c = np.ascontiguousarray(ctr, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    _host_lib().synth_philox_block(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def fill_host(kind, n, seed, stream, first_index=0):
    """n consecutive samples of a stream as a float32 numpy array ("w": weight
    distribution, "x": activation distribution)."""
    rng, e = _params(kind)
    out = np.empty(int(n), dtype=np.float32)
    if n:
        _host_lib().synth_fill_host(out.ctypes.data, int(n), int(seed), int(stream), int(first_index), rng, e)
    return out


def sign_vector(k, seed, stream):
    """k signs (+1 / -1, int8) from the sign bits of a seeded activation
    stream: the rotation's diagonal S of one K width."""
    x = fill_host("x", k, seed, stream)
    return np.where(x < 0, -1, 1).astype(np.int8)


def matrix_rows_host(n_rows_total, k, rows, seed, stream):
    """Selected rows of an n x k weight matrix (row-major element index)."""
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.size, k), dtype=np.float32)
    for i, r in enumerate(rows):
        if not 0 <= r < n_rows_total:
            raise IndexError(r)
        out[i] = fill_host("w", k, seed, stream, int(r) * k)
    return out


def fill_device(ptr, kind, n, seed, stream, first_index=0, cuda_stream=0):
    """Fill n floats at device address ptr with the same values fill_host gives."""
    rng, e = _params(kind)
    rc = _dev_lib().synth_fill_device(ctypes.c_void_p(int(ptr)), int(n), int(seed), int(stream), int(first_index),
                                      rng, e, ctypes.c_void_p(int(cuda_stream)))
    if rc != 0:
        raise RuntimeError(f"synth_fill_device failed with CUDA error {rc}")
