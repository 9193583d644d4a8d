"""CPU checks of the C-ABI library: it loads, exports every symbol the header
declares, its host quantizers produce the oracle's bytes, its host Hadamard
matches the oracle, and invalid arguments are rejected on the host before
any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kq():
    import __graft_entry__

    __graft_entry__.build()
    import quantized_weight_streaming_gb300 as kq

    return kq


def _header_functions():
    text = open(os.path.join(ROOT, "include", "kq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kq_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(kq):
    names = _header_functions()
    assert len(names) >= 25
    lib = ctypes.CDLL(kq.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(kq.SIGNATURES) == names


def test_layout_queries(kq):
    assert kq.kq_block_size("q8_0") == 32 and kq.kq_block_size("pq2_0") == 128
    assert kq.kq_blocks_bytes("q8_0", 1, 128) == 136
    assert kq.kq_blocks_bytes("pq2_0", 10240, 5120) == 13_926_400
    assert kq.kq_scale_stride("q8_0", 2560) == 80
    assert kq.kq_scale_stride("pq2_0", 384) == 8  # 3 blocks, padded to 8
    assert kq.kq_codes_bytes("pq2_0", 2, 512) == 256
    assert kq.kq_scales_bytes("q8_0", 3, 64) == 3 * 8 * 2
    assert kq.kq_codes_bytes("q8_0", 1, 33) == 0  # not a multiple of the block


@pytest.mark.parametrize("seed", [0, 1])
def test_host_q8_0_quantizer_matches_oracle_bytes(kq, seed):
    w = synth.fill_host("w", 96 * 2560, seed, synth.stream_id("test", 0, 200)).reshape(96, 2560)
    assert np.array_equal(kq.kq_quantize_q8_0(w), oracle.q8_0_quantize(w))
    rng = np.random.default_rng(seed)
    wide = (rng.standard_normal((64, 512)) * rng.uniform(1e-6, 50, size=(64, 1))).astype(np.float32)
    wide[3, :32] = 0
    wide[5, 40] = 127 * 0.5  # ties against d = 0.5
    assert np.array_equal(kq.kq_quantize_q8_0(wide), oracle.q8_0_quantize(wide))


@pytest.mark.parametrize("seed", [0, 1])
def test_host_pq2_0_quantizer_matches_oracle_bytes(kq, seed):
    w = synth.fill_host("w", 40 * 5120, seed, synth.stream_id("test", 0, 201)).reshape(40, 5120)
    _, w_rot = oracle.rotate_rows(w)
    assert np.array_equal(kq.kq_quantize_pq2_0(w_rot), oracle.pq2_0_quantize(w_rot))
    rng = np.random.default_rng(seed)
    wide = (rng.standard_normal((16, 1024)) * rng.uniform(1e-6, 50, size=(16, 1))).astype(np.float32)
    wide[2, :128] = 0
    wide[4, :4] = [2.0, 1.0, -1.0, 0.99999994]  # ties at half the scale
    assert np.array_equal(kq.kq_quantize_pq2_0(wide), oracle.pq2_0_quantize(wide))


def test_host_hadamard_matches_oracle(kq):
    # grid inputs: the block sums are exact, so the results are bit-identical
    w = synth.fill_host("w", 8 * 1024, 0, synth.stream_id("test", 0, 202)).reshape(8, 1024)
    _, ref32 = oracle.rotate_rows(w)
    assert np.array_equal(kq.kq_hadamard_blockwise_host(w, 128), ref32)
    # general inputs: within a few fp32 rounding steps
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 4096)).astype(np.float32) * 3
    ref64, _ = oracle.rotate_rows(x, 128)
    got = kq.kq_hadamard_blockwise_host(x, 128)
    assert np.max(np.abs(got - ref64)) <= 2 * np.finfo(np.float32).eps * np.max(np.abs(ref64))
    for block in (1, 2, 64, 1024):
        ref64, _ = oracle.rotate_rows(x, block)
        assert np.max(np.abs(kq.kq_hadamard_blockwise_host(x, block) - ref64)) < 1e-4


@pytest.mark.parametrize("seed", [0, 1])
def test_host_scale4_quantizer_matches_oracle_bytes(kq, seed):
    w = synth.fill_host("w", 64 * 2560, seed, synth.stream_id("test", 0, 207)).reshape(64, 2560)
    assert np.array_equal(kq.kq_quantize_scale4(w), oracle.scale4_quantize(w))
    rng = np.random.default_rng(seed)
    wide = (rng.standard_normal((32, 128)) * rng.uniform(1e-6, 50, size=(32, 1))).astype(np.float32)
    wide[3, :32] = 0
    wide[4, 5], wide[4, 6] = 7.0, -7.0  # a magnitude tie of opposite signs
    wide[4, :5] = 0
    assert np.array_equal(kq.kq_quantize_scale4(wide), oracle.scale4_quantize(wide))
    assert kq.kq_blocks_bytes("scale4", 64, 2560) == 64 * 80 * 18
    assert kq.kq_codes_bytes("scale4", 64, 2560) == 64 * 1280
    assert kq.kq_scale_stride("scale4", 2560) == 80
    lib = kq.lib()
    big = np.full((1, 32), 6e5, dtype=np.float32)
    out = np.full(18, 0xAB, dtype=np.uint8)
    assert lib.kq_quantize_scale4(big.ctypes.data, 1, 32, out.ctypes.data) == kq.KQ_ERR_RANGE
    assert np.all(out == 0xAB)


@pytest.mark.parametrize("seed", [0, 1])
def test_host_ptq1_0_quantizer_matches_oracle_bytes(kq, seed):
    w = synth.fill_host("w", 40 * 1024, seed, synth.stream_id("test", 0, 204)).reshape(40, 1024)
    _, w_rot = oracle.rotate_rows(w)
    assert np.array_equal(kq.kq_quantize_ptq1_0(w_rot), oracle.ptq1_0_quantize(w_rot))
    rng = np.random.default_rng(seed)
    wide = (rng.standard_normal((16, 256)) * rng.uniform(1e-6, 50, size=(16, 1))).astype(np.float32)
    wide[2, :128] = 0
    assert np.array_equal(kq.kq_quantize_ptq1_0(wide), oracle.ptq1_0_quantize(wide))
    assert kq.kq_blocks_bytes("ptq1_0", 40, 1024) == 40 * 8 * 28
    assert kq.kq_codes_bytes("ptq1_0", 40, 1024) == kq.kq_codes_bytes("pq2_0", 40, 1024)


def test_host_signed_rotation_matches_oracle(kq):
    """The page's rotation, n = 1024 with a sign vector, on the host: grid
    inputs make the block sums exact (bit-identical to the oracle), general
    inputs agree within a few fp32 rounding steps."""
    k = 5120
    signs = np.where(np.random.default_rng(11).random(k) < 0.5, -1, 1).astype(np.int8)
    w = synth.fill_host("w", 4 * k, 0, synth.stream_id("test", 0, 203)).reshape(4, k)
    _, ref32 = oracle.rotate_rows(w, 1024, signs=signs)
    assert np.array_equal(kq.kq_rotate_blockwise_host(w, 1024, signs), ref32)
    x = np.random.default_rng(5).standard_normal((3, k)).astype(np.float32)
    ref64, _ = oracle.rotate_rows(x, 1024, signs=signs)
    got = kq.kq_rotate_blockwise_host(x, 1024, signs)
    assert np.max(np.abs(got - ref64)) <= 2 * np.finfo(np.float32).eps * np.max(np.abs(ref64))
    assert np.array_equal(kq.kq_rotate_blockwise_host(x, 128, None), kq.kq_hadamard_blockwise_host(x, 128))
    bad = signs.copy()
    bad[9] = 0
    with pytest.raises(kq.KQError):
        kq.kq_rotate_blockwise_host(x, 1024, bad)


def test_host_errors_leave_output_untouched(kq):
    lib = kq.lib()
    out = np.full(34 * 4, 0xAB, dtype=np.uint8)
    w = np.zeros((1, 48), dtype=np.float32)
    assert lib.kq_quantize_q8_0(w.ctypes.data, 1, 48, out.ctypes.data) == kq.KQ_ERR_SHAPE
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, 77] = np.inf
    assert lib.kq_quantize_q8_0(w.ctypes.data, 1, 128, out.ctypes.data) == kq.KQ_ERR_NONFINITE
    assert lib.kq_quantize_pq2_0(w.ctypes.data, 1, 128, out.ctypes.data) == kq.KQ_ERR_NONFINITE
    w[0, 77] = 1e7
    assert lib.kq_quantize_q8_0(w.ctypes.data, 1, 128, out.ctypes.data) == kq.KQ_ERR_RANGE
    w[0, 77] = 7e4
    assert lib.kq_quantize_pq2_0(w.ctypes.data, 1, 128, out.ctypes.data) == kq.KQ_ERR_RANGE
    assert np.all(out == 0xAB)
    assert "overflows fp16" in lib.kq_last_error().decode()
    assert lib.kq_quantize_q8_0(None, 1, 32, out.ctypes.data) == kq.KQ_ERR_INVALID_ARG
    x = np.zeros((1, 96), dtype=np.float32)
    assert lib.kq_hadamard_blockwise_host(x.ctypes.data, x.ctypes.data, 1, 96, 64) == kq.KQ_ERR_SHAPE
    assert lib.kq_hadamard_blockwise_host(x.ctypes.data, x.ctypes.data, 1, 96, 3) == kq.KQ_ERR_SHAPE


def test_device_entry_points_validate_before_any_cuda_call(kq):
    lib = kq.lib()
    A = 1 << 20  # a 16-byte-aligned fake address; validation must fail before it is used
    bad_k = kq.kq_qmat(kq.KQ_Q8_0, 0, 8, 48, A, A)
    assert lib.kq_gemv_q8_0(ctypes.byref(bad_k), A, A, None, 0, None) == kq.KQ_ERR_SHAPE
    wrong_fmt = kq.kq_qmat(kq.KQ_PQ2_0, 128, 8, 128, A, A)
    assert lib.kq_gemv_q8_0(ctypes.byref(wrong_fmt), A, A, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    no_had = kq.kq_qmat(kq.KQ_PQ2_0, 0, 8, 128, A, A)
    assert lib.kq_gemv_pq2_0(ctypes.byref(no_had), A, A, None, 0, None) == kq.KQ_ERR_UNSUPPORTED
    misaligned = kq.kq_qmat(kq.KQ_Q8_0, 0, 8, 64, A + 4, A)
    assert lib.kq_gemv_q8_0(ctypes.byref(misaligned), A, A, None, 0, None) == kq.KQ_ERR_ALIGNMENT
    good = kq.kq_qmat(kq.KQ_Q8_0, 0, 8, 64, A, A)
    assert lib.kq_gemv_q8_0(ctypes.byref(good), A + 8, A, None, 0, None) == kq.KQ_ERR_ALIGNMENT
    assert lib.kq_gemm_small_m(ctypes.byref(good), A, 65, A, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemm_small_m(ctypes.byref(good), A, 0, A, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemm_splitk(ctypes.byref(good), A, 1, A, -1, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_gemm_tc(ctypes.byref(good), A, 65, A, 0, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemm_tc(ctypes.byref(good), A, 0, A, 0, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemm_tc(ctypes.byref(good), A, 16, A, -1, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_gemm_tc(ctypes.byref(good), None, 16, A, 0, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_gemm_tc(ctypes.byref(good), A + 4, 16, A, 0, None, 0, None) == kq.KQ_ERR_ALIGNMENT
    wide = kq.kq_qmat(kq.KQ_Q8_0, 0, 8, 32800, A, A)
    assert lib.kq_gemm_tc(ctypes.byref(wide), A, 16, A, 0, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemm_tc(ctypes.byref(bad_k), A, 16, A, 0, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemm_tc_workspace_bytes(ctypes.byref(good), 65, 0) == 0
    assert lib.kq_gemv_q8_0(None, A, A, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_dequantize(ctypes.byref(bad_k), A, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_hadamard_blockwise(A, A, 1, 100, 128, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_hadamard_blockwise(A, A, 1, 8192, 8192, None) == kq.KQ_ERR_UNSUPPORTED
    assert lib.kq_prepare(5, A, 1, 32, A, A, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_quantize_pq2_0_device(A, 1, 64, A, A, None) == kq.KQ_ERR_SHAPE
    h = ctypes.c_void_p()
    mixed = (kq.kq_qmat * 2)(good, kq.kq_qmat(kq.KQ_PQ2_0, 128, 8, 128, A, A))
    assert lib.kq_decode_plan_create(mixed, 2, ctypes.byref(h)) in (kq.KQ_ERR_UNSUPPORTED, kq.KQ_ERR_CUDA)
    assert lib.kq_decode_plan_create(mixed, 0, ctypes.byref(h)) == kq.KQ_ERR_SHAPE
    assert lib.kq_decode_step(None, A, A, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_decode_step_host(None, A, A, A, A, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_selftest_bounded_wait(0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_selftest_bounded_wait(1 << 40, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_gemv_workspace_bytes(ctypes.byref(bad_k), 1) == 0
    h1024 = kq.kq_qmat(kq.KQ_PQ2_0, 1024, 8, 1536, A, A)  # k not a multiple of the rotation block
    assert lib.kq_gemv_pq2_0(ctypes.byref(h1024), A, A, None, 0, None) == kq.KQ_ERR_SHAPE
    h512 = kq.kq_qmat(kq.KQ_PQ2_0, 512, 8, 1024, A, A)
    assert lib.kq_gemv_pq2_0(ctypes.byref(h512), A, A, None, 0, None) == kq.KQ_ERR_UNSUPPORTED
    q8_signs = kq.kq_qmat(kq.KQ_Q8_0, 0, 8, 64, A, A, A)
    assert lib.kq_gemv_q8_0(ctypes.byref(q8_signs), A, A, None, 0, None) == kq.KQ_ERR_UNSUPPORTED
    bad_signs = kq.kq_qmat(kq.KQ_PQ2_0, 1024, 8, 1024, A, A, A + 3)
    assert lib.kq_gemv_pq2_0(ctypes.byref(bad_signs), A, A, None, 0, None) == kq.KQ_ERR_ALIGNMENT
    assert lib.kq_rotate_blockwise(A, A, 1, 2048, 1024, A + 1, None) == kq.KQ_ERR_ALIGNMENT
    assert lib.kq_rotate_blockwise(A, A, 1, 1000, 1024, None, None) == kq.KQ_ERR_SHAPE
    s4 = kq.kq_qmat(kq.KQ_SCALE4, 0, 8, 2560, A, A)
    assert lib.kq_gemm_tc(ctypes.byref(s4), A, 65, A, 0, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_gemv_scale4(ctypes.byref(good), A, A, None, 0, None) == kq.KQ_ERR_INVALID_ARG  # a Q8_0 matrix
    s4_bad = kq.kq_qmat(kq.KQ_SCALE4, 0, 8, 48, A, A)
    assert lib.kq_gemv_scale4(ctypes.byref(s4_bad), A, A, None, 0, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_embed(ctypes.byref(good), None, 4, A, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_embed(ctypes.byref(good), A + 4, 4, A, None) == kq.KQ_ERR_ALIGNMENT
    assert lib.kq_embed(ctypes.byref(good), A, -1, A, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_embed(ctypes.byref(good), A, 0, A, None) == kq.KQ_OK  # nothing to do
    wide_pq = kq.kq_qmat(kq.KQ_PQ2_0, 128, 8, 65536, A, A)
    assert lib.kq_embed(ctypes.byref(wide_pq), A, 4, A, None) == kq.KQ_ERR_UNSUPPORTED
    ptq = kq.kq_qmat(kq.KQ_PTQ1_0, 128, 8, 128, A, A)  # a storage format is not a matrix format
    assert lib.kq_gemv_pq2_0(ctypes.byref(ptq), A, A, None, 0, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_stream_read(None, 1024, 4096, 4, A, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_stream_read(A, 1000, 4096, 4, A, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_stream_read(A, 0, 4096, 4, A, None) == kq.KQ_ERR_SHAPE
    assert lib.kq_stream_read(A, 1024, 4100, 4, A, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_stream_read(A, 1024, 512, 4, A, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_stream_read(A, 1024, 4096, 9, A, None) == kq.KQ_ERR_INVALID_ARG
    assert lib.kq_stream_read(A, 1024, 98304, 3, A, None) == kq.KQ_ERR_INVALID_ARG  # ring above 227 KB
    assert lib.kq_stream_read(A + 8, 1024, 4096, 4, A, None) == kq.KQ_ERR_ALIGNMENT


def test_linked_plan_links_validated_before_any_cuda_call(kq):
    """kq_decode_plan_create_linked checks every link on the host first:
    its kind, that the source is an earlier matrix, the stage order, that an
    output is read only by a later stage, k against the source's n (or its
    k for a grouped matvec), a finite alpha and the reserved field."""
    lib = kq.lib()
    A = 1 << 20
    m = lambda n, k: kq.kq_qmat(kq.KQ_Q8_0, 0, n, k, A, A)  # noqa: E731
    h = ctypes.c_void_p()

    def create(mats, links):
        arr = (kq.kq_qmat * len(mats))(*mats)
        la = (kq.kq_link * len(links))(*[kq.kq_link(*lk) for lk in links])
        return lib.kq_decode_plan_create_linked(arr, la, len(mats), ctypes.byref(h))

    P, I, O = 0, 1, 2
    three = [m(256, 256), m(256, 256), m(256, 256)]
    assert create(three, [(P, 0, 0, 1.0, 0), (I, 0, 0, 1.0, 0), (O, 0, 1, 1.0, 0)]) == kq.KQ_ERR_SHAPE  # own stage
    assert create(three, [(P, 1, 0, 1.0, 0), (P, 0, 0, 1.0, 0), (P, 2, 0, 1.0, 0)]) == kq.KQ_ERR_SHAPE  # decreasing
    assert create(three, [(P, 0, 0, 1.0, 0), (O, 1, 2, 1.0, 0), (P, 2, 0, 1.0, 0)]) == kq.KQ_ERR_INVALID_ARG  # later
    assert create(three, [(P, 0, 0, 1.0, 0), (3, 1, 0, 1.0, 0), (P, 2, 0, 1.0, 0)]) == kq.KQ_ERR_INVALID_ARG  # kind
    assert create(three, [(P, 0, 0, 1.0, 0), (O, 1, 0, float("nan"), 0), (P, 2, 0, 1.0, 0)]) == kq.KQ_ERR_INVALID_ARG
    assert create(three, [(P, 0, 0, 1.0, 7), (P, 1, 0, 1.0, 0), (P, 2, 0, 1.0, 0)]) == kq.KQ_ERR_INVALID_ARG  # reserved
    assert create(three, [(P, -1, 0, 1.0, 0), (P, 0, 0, 1.0, 0), (P, 1, 0, 1.0, 0)]) == kq.KQ_ERR_SHAPE  # stage < 0
    wide = [m(256, 256), m(8, 512)]
    assert create(wide, [(P, 0, 0, 1.0, 0), (O, 1, 0, 1.0, 0)]) == kq.KQ_ERR_SHAPE  # k above the source's n
    assert create(wide, [(P, 0, 0, 1.0, 0), (I, 0, 0, 1.0, 0)]) == kq.KQ_ERR_SHAPE  # grouped k differs
    arr = (kq.kq_qmat * 1)(m(256, 256))
    assert lib.kq_decode_plan_create_linked(arr, None, 1, ctypes.byref(h)) == kq.KQ_ERR_INVALID_ARG


def test_status_strings(kq):
    lib = kq.lib()
    for s in range(10):
        assert lib.kq_status_string(s)
    assert lib.kq_status_string(99) == b"unknown status"
    assert lib.kq_version() == 2
