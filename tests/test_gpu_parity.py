"""GPU parity of the CUDA path against the FP64 oracle, through the C ABI.

Bars: integer and byte work (codes, scales, dequantized values, the
generator, the FP64 weight rotation) bit-exact; floating-point outputs within
|y - y_oracle| <= 1e-4 * sum_j |w_ij x_j| per row; integer-valued cases at
tolerance 0."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402

TOL = 1e-4


@pytest.fixture(scope="module")
def kq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import quantized_weight_streaming_gb300 as kq

    torch.cuda.set_device(0)
    kq.kq_device_status(True)
    yield kq
    assert kq.kq_device_status(True) == kq.KQ_OK


@pytest.fixture(scope="module")
def wl(kq):
    import workloads

    return workloads


@pytest.fixture(params=["mma_sync", "tcgen05"])
def consumer(request, kq):
    """Runs a PQ2_0 one-row test under each consumer (kq_set_pq2_0_consumer);
    cases the setting does not touch (other formats, tcgen05 GEMM paths,
    linked plans) run once, under the default."""
    params = request.node.callspec.params
    untouched = (params.get("fmt", "pq2_0") != "pq2_0" or params.get("config", "bonsai_27b_pq2_0_step").startswith("qwen")
                 or params.get("path", "gemv") != "gemv" or params.get("linked", False))
    if request.param == "tcgen05" and untouched:
        pytest.skip("the consumer setting does not apply to this case")
    kq.kq_set_pq2_0_consumer(kq.KQ_PQ2_0_TCGEN05 if request.param == "tcgen05" else kq.KQ_PQ2_0_MMA_SYNC)
    yield request.param
    kq.kq_set_pq2_0_consumer(kq.KQ_PQ2_0_MMA_SYNC)


def _sync_ok(kq):
    torch.cuda.synchronize()
    assert kq.kq_device_status(True) == kq.KQ_OK


def _planes_as_blocks(kq, W):
    """Device planes -> AoS blocks (host: fp16 scale, then the code bytes), for byte comparison."""
    bs = kq.kq_block_size(W.fmt)
    nb = W.k // bs
    cb = 16 if W.fmt == kq.KQ_SCALE4 else 32
    codes = W.codes.cpu().numpy().reshape(W.n, nb, cb)
    ss = kq.kq_scale_stride(W.fmt, W.k)
    scales = W.scales.cpu().numpy().view(np.uint16).reshape(W.n, ss)
    assert not scales[:, nb:].any()  # padding is zero
    out = np.empty((W.n, nb, 2 + cb), dtype=np.uint8)
    out[:, :, 0] = scales[:, :nb] & 0xFF
    out[:, :, 1] = scales[:, :nb] >> 8
    out[:, :, 2:] = codes
    return out


def _run_gemv(kq, W, x, splits=0, m=1):
    y = torch.empty(m * W.n, dtype=torch.float32, device="cuda")
    nbytes = kq.kq_gemm_splitk_workspace_bytes(W, m, splits)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    if splits == 0 and m == 1:
        {kq.KQ_PQ2_0: kq.kq_gemv_pq2_0, kq.KQ_Q8_0: kq.kq_gemv_q8_0, kq.KQ_SCALE4: kq.kq_gemv_scale4}[W.fmt](W, x, y, ws)
    else:
        kq.kq_gemm_splitk(W, x, m, y, splits, ws)
    _sync_ok(kq)
    return y.cpu().numpy().reshape(m, W.n) if m > 1 else y.cpu().numpy()


# ----------------------------------------------------------------------------
# generator, rotation, quantizers
# ----------------------------------------------------------------------------

def test_device_generator_matches_host(kq):
    for kind, n, first in (("w", 1_000_003, 0), ("x", 77_777, 12345)):
        s = synth.stream_id("test", 0, 300)
        d = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.fill_device(d.data_ptr(), kind, n, 5, s, first)
        torch.cuda.synchronize()
        assert np.array_equal(d.cpu().numpy(), synth.fill_host(kind, n, 5, s, first))


def test_device_hadamard_bit_identical_to_host_and_oracle(kq):
    w = synth.fill_host("w", 64 * 1024, 1, synth.stream_id("test", 0, 301)).reshape(64, 1024)
    d = torch.from_numpy(w).cuda()
    out = torch.empty_like(d)
    kq.kq_hadamard_blockwise(d, out, 64, 1024, 128)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got, kq.kq_hadamard_blockwise_host(w, 128))
    assert np.array_equal(got, oracle.rotate_rows(w)[1])  # grid inputs: exact sums
    rng = np.random.default_rng(0)
    g = (rng.standard_normal((8, 2048)) * 10).astype(np.float32)
    dg = torch.from_numpy(g).cuda()
    for block in (2, 64, 128, 256, 2048):
        o = torch.empty_like(dg)
        kq.kq_hadamard_blockwise(dg, o, 8, 2048, block)
        torch.cuda.synchronize()
        assert np.array_equal(o.cpu().numpy(), kq.kq_hadamard_blockwise_host(g, block)), block
    kq.kq_hadamard_blockwise(dg, dg, 8, 2048, 128)  # in place
    torch.cuda.synchronize()
    assert np.array_equal(dg.cpu().numpy(), kq.kq_hadamard_blockwise_host(g, 128))


@pytest.mark.parametrize("fmt,n,k", [("q8_0", 1024, 2560), ("pq2_0", 10240, 5120), ("q8_0", 33, 96),
                                     ("pq2_0", 17, 384), ("scale4", 9728, 2560), ("scale4", 33, 96)])
def test_device_quantizer_and_prepare_bit_exact(kq, wl, fmt, n, k):
    s = synth.stream_id("test", 0, 302)
    W = wl.build_matrix(fmt, n, k, 3, s)
    _sync_ok(kq)
    w = synth.fill_host("w", n * k, 3, s).reshape(n, k)
    if fmt == "q8_0":
        ref = oracle.q8_0_quantize(w)
    elif fmt == "scale4":
        ref = oracle.scale4_quantize(w)
    else:
        ref = oracle.pq2_0_quantize(oracle.rotate_rows(w)[1])
    assert np.array_equal(_planes_as_blocks(kq, W), ref)
    # debug dequantizer is bit-exact against the oracle's dequantizer
    deq = torch.empty(n * k, dtype=torch.float32, device="cuda")
    kq.kq_dequantize(W, deq)
    _sync_ok(kq)
    ref_deq = {"q8_0": oracle.q8_0_dequant, "scale4": oracle.scale4_dequant, "pq2_0": oracle.pq2_0_dequant}[fmt](ref, n, k)
    assert np.array_equal(deq.cpu().numpy().reshape(n, k), ref_deq)
    # AoS blocks from the host quantizer, repacked on the device, give the same planes
    W2 = kq.QMatrix(fmt, n, k)
    blocks = torch.from_numpy(np.ascontiguousarray(ref).reshape(-1)).cuda()
    kq.kq_prepare(W2, blocks)
    _sync_ok(kq)
    assert torch.equal(W2.codes, W.codes) and torch.equal(W2.scales, W.scales)


@pytest.mark.parametrize("n,k", [(300, 5120), (17, 1024), (1000, 128)])
def test_ptq1_0_transcode_to_pq2_0_planes(kq, wl, n, k):
    """PTQ1_0 blocks (the page's base-3 download format) transcoded on the
    device give exactly the PQ2_0 planes of the same rotated weights; the
    GEMV on them matches the oracle."""
    sid = synth.stream_id("test", 0, 460 + n)
    w = synth.fill_host("w", n * k, 8, sid).reshape(n, k)
    _, w_rot = oracle.rotate_rows(w)
    ptq = oracle.ptq1_0_quantize(w_rot)
    W = kq.QMatrix("pq2_0", n, k)
    kq.kq_prepare(W, torch.from_numpy(ptq.reshape(-1)).cuda(), block_fmt="ptq1_0")
    _sync_ok(kq)
    assert np.array_equal(_planes_as_blocks(kq, W), oracle.pq2_0_quantize(w_rot))
    x = synth.fill_host("x", k, 8, synth.stream_id("test", 1, 461))
    _, _, y_ref, absdot = oracle.reference("pq2_0", w, x)
    ok, worst = oracle.within_bound(_run_gemv(kq, W, torch.from_numpy(x).cuda()), y_ref, absdot, TOL)
    assert ok, worst


def test_device_quantizer_flags_nonfinite_and_range(kq):
    W = kq.QMatrix("q8_0", 2, 64)
    w = torch.zeros(128, dtype=torch.float32, device="cuda")
    w[5] = float("nan")
    kq.kq_quantize_q8_0_device(W, w)
    assert kq.kq_device_status(True) == kq.KQ_ERR_NONFINITE
    w[5] = 1e7
    kq.kq_quantize_q8_0_device(W, w)
    assert kq.kq_device_status(True) == kq.KQ_ERR_RANGE
    assert kq.kq_device_status(True) == kq.KQ_OK


# ----------------------------------------------------------------------------
# GEMV parity
# ----------------------------------------------------------------------------

SHAPES = [
    ("q8_0", 1024, 2560),    # Q8_0 GEMV workload, full size
    ("pq2_0", 10240, 5120),  # PQ2_0 GEMV workload, full size
    ("q8_0", 1, 32), ("q8_0", 17, 96), ("q8_0", 72, 2592), ("q8_0", 33, 9728), ("q8_0", 5, 4096),
    ("pq2_0", 1, 128), ("pq2_0", 15, 384), ("pq2_0", 72, 5248), ("pq2_0", 31, 17408), ("pq2_0", 48, 6144),
    ("scale4", 1024, 2560), ("scale4", 9728, 2560), ("scale4", 2560, 9728), ("scale4", 1, 32), ("scale4", 17, 96),
    ("scale4", 300, 4128), ("scale4", 33, 16384),
]


@pytest.mark.parametrize("fmt,n,k", SHAPES)
def test_gemv_matches_oracle(kq, consumer, wl, fmt, n, k):
    sw, sx = synth.stream_id("test", 0, 310), synth.stream_id("test", 1, 310)
    W = wl.build_matrix(fmt, n, k, 0, sw)
    x = wl.build_activation(k, 0, sx)
    y = _run_gemv(kq, W, x)
    w = synth.fill_host("w", n * k, 0, sw).reshape(n, k)
    xh = synth.fill_host("x", k, 0, sx)
    _, _, y_ref, absdot = oracle.reference(fmt, w, xh)
    ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
    assert ok, f"worst error/bound {worst}"
    # deterministic: a second call gives the same bits
    assert np.array_equal(_run_gemv(kq, W, x), y)


@pytest.mark.parametrize("fmt", ["q8_0", "pq2_0", "scale4"])
def test_gemv_at_k_32768(kq, consumer, wl, fmt):
    """The largest K the tests use for a single GEMV (above a plan's staging
    limit, so it is split): every row against the oracle."""
    n, k = 40, 32768
    sw, sx = synth.stream_id("test", 0, 311), synth.stream_id("test", 1, 311)
    W = wl.build_matrix(fmt, n, k, 0, sw)
    y = _run_gemv(kq, W, wl.build_activation(k, 0, sx))
    _, _, y_ref, absdot = oracle.reference(fmt, synth.fill_host("w", n * k, 0, sw).reshape(n, k),
                                           synth.fill_host("x", k, 0, sx))
    ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
    assert ok, worst


@pytest.mark.parametrize("fmt,limit,block", [("q8_0", 18432, 32), ("pq2_0", 18432, 128), ("scale4", 16384, 32)])
def test_decode_plan_at_its_staging_limit(kq, consumer, wl, fmt, limit, block):
    """A plan accepts a matrix whose K is exactly the staging limit (every
    row checked) and refuses one block more with KQ_ERR_UNSUPPORTED."""
    n = 70
    sw, sx = synth.stream_id("test", 0, 312), synth.stream_id("test", 1, 312)
    W = wl.build_matrix(fmt, n, limit, 2, sw)
    plan = kq.DecodePlan([W])
    x = synth.fill_host("x", limit, 2, sx)
    y = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    plan.step(torch.from_numpy(x).cuda(), y)
    _sync_ok(kq)
    _, _, y_ref, absdot = oracle.reference(fmt, synth.fill_host("w", n * limit, 2, sw).reshape(n, limit), x)
    ok, worst = oracle.within_bound(y.cpu().numpy(), y_ref, absdot, TOL)
    assert ok, worst
    plan.close()
    big = wl.build_matrix(fmt, 8, limit + block, 2, sw)
    with pytest.raises(kq.KQError) as e:
        kq.DecodePlan([big])
    assert e.value.status == kq.KQ_ERR_UNSUPPORTED


def test_q8_0_exact_integer_case_tolerance_zero(kq):
    # integer codes, power-of-two scales, small integer activations: every
    # partial sum is an exact fp32 value, so the result must match exactly
    rng = np.random.default_rng(11)
    n, k = 72, 2816  # ragged rows and a K that is not a multiple of the chunk
    q = rng.integers(-127, 128, size=(n, k))
    q[:, ::32] = 127
    w = (q * 2.0**-5).astype(np.float32)
    x = rng.integers(-8, 9, size=k).astype(np.float32)
    blocks, _, y_ref, _ = oracle.q8_0_reference(w, x)
    W = kq.QMatrix("q8_0", n, k)
    kq.kq_prepare(W, torch.from_numpy(blocks.reshape(-1)).cuda())
    y = _run_gemv(kq, W, torch.from_numpy(x).cuda())
    assert np.array_equal(y.astype(np.float64), y_ref)
    assert np.array_equal(y_ref, (q @ x.astype(np.int64)) * 2.0**-5)


def test_scale4_exact_integer_case_tolerance_zero(kq):
    """Codes 0..15 with a 0 in every block (so d = 2^-5 exactly), small
    integer activations: every product and partial sum is exact in fp32, the
    zero point included, so the output must equal the oracle's exactly."""
    rng = np.random.default_rng(14)
    n, k = 300, 4128  # ragged rows, K not a multiple of the 512-weight tile row
    q = rng.integers(0, 16, size=(n, k))
    q[:, ::32] = 0
    w = ((q - 8) * 2.0**-5).astype(np.float32)
    x = rng.integers(-8, 9, size=k).astype(np.float32)
    blocks, _, y_ref, _ = oracle.scale4_reference(w, x)
    W = kq.QMatrix("scale4", n, k)
    kq.kq_prepare(W, torch.from_numpy(blocks.reshape(-1)).cuda())
    y = _run_gemv(kq, W, torch.from_numpy(x).cuda())
    assert np.array_equal(y.astype(np.float64), y_ref)
    assert np.array_equal(y_ref, ((q - 8) @ x.astype(np.int64)) * 2.0**-5)
    y3 = _run_gemv(kq, W, torch.from_numpy(x).cuda(), splits=3)
    assert np.array_equal(y3.astype(np.float64), y_ref)


def test_pq2_0_nonzero_mean_activation(kq, consumer, wl):
    n, k = 96, 5120
    sw = synth.stream_id("test", 0, 311)
    W = wl.build_matrix("pq2_0", n, k, 0, sw)
    xh = synth.fill_host("x", k, 0, synth.stream_id("test", 1, 311)) + np.float32(4.0)
    y = _run_gemv(kq, W, torch.from_numpy(xh).cuda())
    w = synth.fill_host("w", n * k, 0, sw).reshape(n, k)
    _, _, y_ref, absdot = oracle.pq2_0_reference(w, xh)
    ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
    assert ok, worst


def test_pq2_0_activation_scale_extremes(kq, consumer, wl):
    # per-block exponent normalisation: tiny and huge activations keep precision
    n, k = 32, 1024
    sw = synth.stream_id("test", 0, 312)
    W = wl.build_matrix("pq2_0", n, k, 0, sw)
    w = synth.fill_host("w", n * k, 0, sw).reshape(n, k)
    base = synth.fill_host("x", k, 0, synth.stream_id("test", 1, 312))
    for scale in (2.0**-60, 2.0**-20, 1.0, 2.0**40):
        xh = (base * np.float32(scale)).astype(np.float32)
        xh[:128] *= np.float32(2.0**10)  # blocks of very different magnitude
        y = _run_gemv(kq, W, torch.from_numpy(xh).cuda())
        _, _, y_ref, absdot = oracle.pq2_0_reference(w, xh)
        ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
        assert ok, (scale, worst)


@pytest.mark.parametrize("n,k", [(1023, 4096), (8, 64), (2049, 2560), (5120, 4096)])
def test_q8_0_one_launch_gemv(kq, wl, n, k):
    """A small Q8_0 matrix at one row runs in one launch with no K split: it
    asks for no workspace, is deterministic and within the bound, and so is
    the split streaming path (explicit split counts) on the same inputs.  The
    shapes: k at the path's limit of 4096, a single CTA, rows not a multiple
    of the CTA's 8, and the largest matrix the path takes (20 MB of codes)."""
    sw, sx = synth.stream_id("test", 0, 315), synth.stream_id("test", 1, 315)
    W = wl.build_matrix("q8_0", n, k, 2, sw)
    x = wl.build_activation(k, 2, sx)
    assert kq.kq_gemv_workspace_bytes(W, 1) == 0
    w = synth.fill_host("w", n * k, 2, sw).reshape(n, k)
    _, _, y_ref, absdot = oracle.reference("q8_0", w, synth.fill_host("x", k, 2, sx))
    y = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    kq.kq_gemv_q8_0(W, x, y, None)  # no workspace at all
    _sync_ok(kq)
    y = y.cpu().numpy()
    ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
    assert ok, worst
    assert np.array_equal(_run_gemv(kq, W, x), y)
    for splits in (1, 2):
        ys = _run_gemv(kq, W, x, splits=splits)
        ok, worst = oracle.within_bound(ys, y_ref, absdot, TOL)
        assert ok, (splits, worst)


@pytest.mark.parametrize("fmt,n,k", [("q8_0", 200, 9728), ("pq2_0", 120, 20480), ("pq2_0", 64, 5120)])
def test_split_k(kq, consumer, wl, fmt, n, k):
    sw, sx = synth.stream_id("test", 0, 320), synth.stream_id("test", 1, 320)
    W = wl.build_matrix(fmt, n, k, 1, sw)
    x = wl.build_activation(k, 1, sx)
    w = synth.fill_host("w", n * k, 1, sw).reshape(n, k)
    _, _, y_ref, absdot = oracle.reference(fmt, w, synth.fill_host("x", k, 1, sx))
    outs = {}
    for splits in (1, 2, 3, 0):
        if splits == 1 and k > 18432:
            continue
        y = _run_gemv(kq, W, x, splits=splits)
        ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
        assert ok, (splits, worst)
        assert np.array_equal(_run_gemv(kq, W, x, splits=splits), y)  # same plan, same bits
        outs[splits] = y


def test_workspace_too_small_is_rejected(kq, wl):
    W = wl.build_matrix("pq2_0", 16, 20480, 0, synth.stream_id("test", 0, 321))
    x = wl.build_activation(20480, 0, synth.stream_id("test", 1, 321))
    y = torch.full((16,), 7.0, device="cuda")
    need = kq.kq_gemv_workspace_bytes(W)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kq.KQError) as e:
        kq.kq_gemv_pq2_0(W, x, y, ws)
    assert e.value.status == kq.KQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


# ----------------------------------------------------------------------------
# small-M GEMM
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,n,k", [("q8_0", 9728, 2560), ("pq2_0", 17408, 5120), ("q8_0", 40, 288),
                                     ("pq2_0", 24, 1152), ("scale4", 9728, 2560), ("scale4", 40, 544)])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 16, 64])
def test_small_m_matches_oracle(kq, wl, fmt, n, k, m):
    if n * k > 50_000_000 and m not in (1, 4, 16, 64):
        pytest.skip("full-size matrices run only at the workload's M values")
    sw, sx = synth.stream_id("test", 0, 330), synth.stream_id("test", 1, 330 + m)
    W = wl.build_matrix(fmt, n, k, 2, sw)
    X = wl.build_activation(k, 2, sx, rows=m)
    Y = torch.empty(m * n, dtype=torch.float32, device="cuda")
    nbytes = kq.kq_gemv_workspace_bytes(W, m)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    kq.kq_gemm_small_m(W, X, m, Y, ws)
    _sync_ok(kq)
    Y = Y.cpu().numpy().reshape(m, n)
    rows = np.arange(n) if n * k <= 50_000_000 else np.unique(np.r_[0, n - 1, np.arange(7, n, 997)])
    w = synth.matrix_rows_host(n, k, rows, 2, sw)
    Xh = synth.fill_host("x", m * k, 2, sx).reshape(m, k)
    if fmt == "pq2_0":
        deq = oracle.pq2_0_dequant(oracle.pq2_0_quantize(oracle.rotate_rows(w)[1]), rows.size, k)
        X64 = oracle.rotate_rows(Xh)[0]
    elif fmt == "scale4":
        deq = oracle.scale4_dequant(oracle.scale4_quantize(w), rows.size, k)
        X64 = Xh.astype(np.float64)
    else:
        deq = oracle.q8_0_dequant(oracle.q8_0_quantize(w), rows.size, k)
        X64 = Xh.astype(np.float64)
    for i in range(m):
        y_ref, absdot = oracle.gemv(deq, X64[i])
        ok, worst = oracle.within_bound(Y[i, rows], y_ref, absdot, TOL)
        assert ok, (i, worst)


# ----------------------------------------------------------------------------
# small-M GEMM on the tensor cores (tcgen05)
# ----------------------------------------------------------------------------

def _small_m_reference(fmt, n, k, m, seed, sw, sx, rows):
    """Oracle dequantized rows and (rotated for PQ2_0) FP64 activations."""
    w = synth.matrix_rows_host(n, k, rows, seed, sw)
    Xh = synth.fill_host("x", m * k, seed, sx).reshape(m, k)
    if fmt == "pq2_0":
        deq = oracle.pq2_0_dequant(oracle.pq2_0_quantize(oracle.rotate_rows(w)[1]), rows.size, k)
        X64 = oracle.rotate_rows(Xh)[0]
    elif fmt == "scale4":
        deq = oracle.scale4_dequant(oracle.scale4_quantize(w), rows.size, k)
        X64 = Xh.astype(np.float64)
    else:
        deq = oracle.q8_0_dequant(oracle.q8_0_quantize(w), rows.size, k)
        X64 = Xh.astype(np.float64)
    return deq, X64


def _run_tc(kq, W, X, m, splits):
    Y = torch.full((m * W.n,), 7.0, dtype=torch.float32, device="cuda")
    nbytes = kq.kq_gemm_tc_workspace_bytes(W, m, splits)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    kq.kq_gemm_tc(W, X, m, Y, splits, ws)
    _sync_ok(kq)
    return Y.cpu().numpy().reshape(m, W.n)


@pytest.mark.parametrize("fmt,n,k", [("q8_0", 300, 2080), ("scale4", 300, 2080), ("pq2_0", 200, 1152)])
@pytest.mark.parametrize("m", [1, 3, 16, 33])
def test_full_mantissa_activations(kq, wl, consumer, fmt, n, k, m):
    """Activations with full 24-bit mantissas (not the generator's 2^-16
    grid), each 32-block scaled by its own power of two in 2^-12 .. 2^12:
    the fp16 high/low split of the tensor-core paths (m = 16, 33), the
    per-block normalisation of the streaming consumers (m = 1, 3) and the
    transform's rounding all see values they do not hold exactly."""
    if m != 1 and consumer == "tcgen05":
        pytest.skip("the consumer setting applies to one activation row")
    sw = synth.stream_id("test", 0, 340)
    W = wl.build_matrix(fmt, n, k, 3, sw)
    w = synth.fill_host("w", n * k, 3, sw).reshape(n, k)
    rng = np.random.default_rng(340 + m)
    X = rng.standard_normal((m, k)).astype(np.float32)
    X *= np.exp2(rng.integers(-12, 13, size=(m, k // 32))).repeat(32, axis=1).astype(np.float32)
    assert np.count_nonzero(X.view(np.uint32) & 0xFF) > 0.9 * X.size  # low mantissa bits in use
    Xd = torch.from_numpy(X.reshape(-1)).cuda()
    if m >= 16:
        Y = _run_tc(kq, W, Xd, m, 0)
    else:
        Y = _run_gemv(kq, W, Xd, splits=0 if m == 1 else 2, m=m).reshape(m, n)
    for i in range(m):
        _, _, y_ref, absdot = oracle.reference(fmt, w, X[i])
        ok, worst = oracle.within_bound(Y[i], y_ref, absdot, TOL)
        assert ok, (i, worst)


@pytest.mark.parametrize("fmt,n,k", [("q8_0", 300, 2080), ("pq2_0", 200, 1152), ("q8_0", 128, 128),
                                     ("pq2_0", 1, 128), ("q8_0", 1000, 4096), ("pq2_0", 520, 5120),
                                     ("scale4", 300, 2080), ("scale4", 1000, 4096), ("scale4", 1, 32)])
@pytest.mark.parametrize("m", [1, 5, 16, 33, 64])
@pytest.mark.parametrize("splits", [0, 3])
def test_tc_gemm_matches_oracle(kq, wl, fmt, n, k, m, splits):
    # ragged row tiles (n % 128), a ragged last K chunk (Q8_0 k = 2080), M not a
    # multiple of 8, forced and automatic K splits
    sw, sx = synth.stream_id("test", 0, 340), synth.stream_id("test", 1, 340 + m)
    W = wl.build_matrix(fmt, n, k, 4, sw)
    X = wl.build_activation(k, 4, sx, rows=m)
    Y = _run_tc(kq, W, X, m, splits)
    rows = np.arange(n)
    deq, X64 = _small_m_reference(fmt, n, k, m, 4, sw, sx, rows)
    for i in range(m):
        y_ref, absdot = oracle.gemv(deq, X64[i])
        ok, worst = oracle.within_bound(Y[i], y_ref, absdot, TOL)
        assert ok, (i, worst)
    # same plan, same bits
    assert np.array_equal(_run_tc(kq, W, X, m, splits), Y)


def test_tc_scale4_exact_integer_case_tolerance_zero(kq):
    """The tcgen05 path on scale4 codes with a 0 in every block (d = 2^-5)
    and small integer activations: every product and sum is exact, so the
    output equals the oracle's exactly (the codes enter the tensor core as the
    exact (q - 8) * 2^(s - 24))."""
    rng = np.random.default_rng(16)
    n, k, m = 300, 2080, 16
    q = rng.integers(0, 16, size=(n, k))
    q[:, ::32] = 0
    w = ((q - 8) * 2.0**-5).astype(np.float32)
    X = rng.integers(-8, 9, size=(m, k)).astype(np.float32)
    blocks = oracle.scale4_quantize(w)
    W = kq.QMatrix("scale4", n, k)
    kq.kq_prepare(W, torch.from_numpy(blocks.reshape(-1)).cuda())
    Y = _run_tc(kq, W, torch.from_numpy(X.reshape(-1)).cuda(), m, 0)
    want = ((q - 8) @ X.T.astype(np.int64)).T * 2.0**-5
    assert np.array_equal(Y.astype(np.float64), want)


def test_tc_q8_0_exact_integer_case_tolerance_zero(kq):
    # power-of-two scales make fp16(q*d) exact, small integer activations make
    # the high part exact and the low part zero, and every partial sum is an
    # exact fp32 value: the tensor-core result must equal the exact product,
    # which pins the tile layouts (any transposed, permuted or shifted operand
    # changes it)
    rng = np.random.default_rng(12)
    n, k, m = 200, 2848, 16
    q = rng.integers(-127, 128, size=(n, k))
    q[:, ::32] = 127
    w = (q * 2.0**-5).astype(np.float32)
    X = rng.integers(-8, 9, size=(m, k)).astype(np.float32)
    X[3] = 0.0  # an all-zero activation row
    blocks = oracle.q8_0_quantize(w)
    W = kq.QMatrix("q8_0", n, k)
    kq.kq_prepare(W, torch.from_numpy(blocks.reshape(-1)).cuda())
    for splits in (1, 0, 5):
        Y = _run_tc(kq, W, torch.from_numpy(X.reshape(-1)).cuda(), m, splits)
        assert np.array_equal(Y.astype(np.float64), (X.astype(np.int64) @ q.T) * 2.0**-5), splits


def _single_weight_pq2_0(kq, n, k, d=2.0**-3):
    """PQ2_0 matrix whose row r holds one nonzero ternary weight, at column
    (r * 37) % k (all other codes 1, value 0); returns (W, codes)."""
    blocks = np.zeros((n, k // 128, 34), dtype=np.uint8)
    dbits = np.array([d], dtype=np.float16).view(np.uint16)[0]
    blocks[:, :, 0] = dbits & 0xFF
    blocks[:, :, 1] = dbits >> 8
    codes = np.ones((n, k), dtype=np.uint8)
    cols = (np.arange(n) * 37) % k
    codes[np.arange(n), cols] = np.where(np.arange(n) % 3, 2, 0)
    for j in range(k):
        blocks[:, j // 128, 2 + (j % 128) // 4] |= (codes[:, j] << (2 * (j % 4))).astype(np.uint8)
    W = kq.QMatrix("pq2_0", n, k)
    kq.kq_prepare(W, torch.from_numpy(blocks.reshape(-1)).cuda())
    return W, codes, cols


@pytest.mark.parametrize("path", ["gemv", "tc"])
def test_pq2_0_single_weight_rows(kq, consumer, path):
    # row r holds one nonzero ternary weight: y[r] = +-d x'[col r], so the
    # bound 1e-4 * sum |w x'| is 1e-4 * d |x'[col r]|.  This pins the code
    # pairing and B permutation, and fails a kernel that forms sum c x' and
    # subtracts sum x' afterwards (the accumulator's rounding of the cancelled
    # terms is far above the bound).  The rotated activations x' are integers
    # of magnitude 16..64 (x = R x' in FP64, rounded to fp32).
    n, k = 200, 5120
    m = 1 if path == "gemv" else 16
    W, codes, cols = _single_weight_pq2_0(kq, n, k)
    rng = np.random.default_rng(13)
    xr = (rng.integers(16, 65, size=(m, k)) * rng.choice([-1, 1], size=(m, k))).astype(np.float32)
    X = oracle.rotate_rows(xr)[1]  # R is its own inverse
    if path == "gemv":
        Y = _run_gemv(kq, W, torch.from_numpy(X.reshape(-1)).cuda()).reshape(1, n)
    else:
        Y = _run_tc(kq, W, torch.from_numpy(X.reshape(-1)).cuda(), m, 1)
    Xr = oracle.rotate_rows(X)[0]
    sign = codes[np.arange(n), cols].astype(np.float64) - 1
    expect = Xr[:, cols] * 2.0**-3 * sign
    assert np.all(np.abs(Y - expect) <= TOL * np.abs(expect)), np.max(np.abs(Y - expect) / (TOL * np.abs(expect)))


def test_tc_workspace_too_small_is_rejected(kq, wl):
    W = wl.build_matrix("q8_0", 256, 1024, 0, synth.stream_id("test", 0, 341))
    X = wl.build_activation(1024, 0, synth.stream_id("test", 1, 341), rows=16)
    Y = torch.full((16 * 256,), 7.0, dtype=torch.float32, device="cuda")
    need = kq.kq_gemm_tc_workspace_bytes(W, 16, 2)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kq.KQError) as e:
        kq.kq_gemm_tc(W, X, 16, Y, 2, ws)
    assert e.value.status == kq.KQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)


# ----------------------------------------------------------------------------
# decode-step driver
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("nbytes,stage_bytes,stages", [(16, 1024, 1), (1040, 1024, 2), (5_000_000 + 48, 34816, 4),
                                                      (3 * 98304 + 16, 98304, 2), (300_000_016, 69632, 2)])
def test_stream_read_control_xor(kq, nbytes, stage_bytes, stages):
    """The read-only control kernel reads every byte once: the XOR of all
    32-bit words is integer work, compared bit-exactly with numpy's."""
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    kq.kq_stream_read(src, nbytes, sink, stage_bytes=stage_bytes, stages=stages)
    _sync_ok(kq)
    want = np.bitwise_xor.reduce(src.cpu().numpy().view(np.uint32))
    assert int(sink[0].item()) & 0xFFFFFFFF == int(want)
    assert not sink[1:].any()


def test_decode_plan_small_mixed_shapes(kq, consumer, wl):
    spec = [(16, 256), (33, 1024), (1, 5120), (300, 2048), (17, 17408), (64, 128)]
    for fmt in ("q8_0", "pq2_0", "scale4"):
        mats, xs, host = [], [], []
        for i, (n, k) in enumerate(spec):
            if fmt == "scale4" and k > 16384:
                continue  # beyond the SCALE4 plan's staging limit
            sw, sx = synth.stream_id("test", 0, 340 + i), synth.stream_id("test", 1, 340 + i)
            mats.append(wl.build_matrix(fmt, n, k, 4, sw))
            xs.append(synth.fill_host("x", k, 4, sx))
            host.append(synth.fill_host("w", n * k, 4, sw).reshape(n, k))
        plan = kq.DecodePlan(mats)
        x = torch.from_numpy(np.concatenate(xs)).cuda()
        y = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
        plan.step(x, y)
        _sync_ok(kq)
        yh = y.cpu().numpy()
        off = 0
        for W, w, xh in zip(mats, host, xs):
            _, _, y_ref, absdot = oracle.reference(fmt, w, xh)
            ok, worst = oracle.within_bound(yh[off:off + W.n], y_ref, absdot, TOL)
            assert ok, (fmt, W.n, W.k, worst)
            # same tiles and one split, as the single GEMV with one split: the same bits
            assert np.array_equal(yh[off:off + W.n], _run_gemv(kq, W, torch.from_numpy(xh).cuda(), splits=1))
            off += W.n
        y2 = torch.empty_like(y)
        plan.step(x, y2)
        _sync_ok(kq)
        assert torch.equal(y, y2)
        plan.close()


# ----------------------------------------------------------------------------
# embedding lookup (gather + dequantize + inverse rotation)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,vocab,dim,had", [("q8_0", 1000, 2560, 0), ("scale4", 700, 2080, 0),
                                               ("pq2_0", 600, 5120, 128), ("pq2_0", 300, 5120, 1024)])
def test_embed_matches_oracle(kq, wl, fmt, vocab, dim, had):
    sid = synth.stream_id("test", 0, 480 + dim % 89)
    sh, sd = (wl.build_signs(dim, 4, synth.stream_id("test", 1, 481)) if had == 1024 else (None, None))
    E = wl.build_matrix(fmt, vocab, dim, 10, sid, had_block=(1024 if had == 1024 else None), signs=sd)
    ids = np.array([0, vocab - 1, 5, 5, 123, 77, vocab // 2], dtype=np.int32)
    out = torch.empty(len(ids) * dim, dtype=torch.float32, device="cuda")
    kq.kq_embed(E, torch.from_numpy(ids).cuda(), len(ids), out)
    _sync_ok(kq)
    got = out.cpu().numpy().reshape(len(ids), dim).astype(np.float64)
    e = synth.matrix_rows_host(vocab, dim, np.arange(vocab), 10, sid)
    if fmt == "pq2_0":
        blocks = oracle.pq2_0_quantize(oracle.rotate_rows(e, had, signs=sh)[1])
    else:
        blocks = (oracle.q8_0_quantize if fmt == "q8_0" else oracle.scale4_quantize)(e)
    want, blk = oracle.embed_reference(fmt, blocks, vocab, dim, ids, had if had else 128, sh)
    if fmt != "pq2_0":
        assert np.array_equal(got, want)  # a dequantized row is exact
    else:  # an fp32 transform: (log2 n + 3) 2^-24 sum_blk |z| / sqrt(n) per element
        n = had
        assert np.all(np.abs(got - want) <= (np.log2(n) + 3) * 2.0**-24 * blk / np.sqrt(n) + 1e-30)
        # the rows are the original (unrotated) embeddings up to the quantization of R e
        assert np.corrcoef(got[0], e[0])[0, 1] > 0.6  # ternary codes of Gaussian rows: about 0.73


def test_embed_out_of_range_ids(kq, wl):
    E = wl.build_matrix("q8_0", 10, 64, 1, synth.stream_id("test", 0, 485))
    ids = torch.tensor([3, -1, 10, 9], dtype=torch.int32, device="cuda")
    out = torch.full((4 * 64,), 7.0, dtype=torch.float32, device="cuda")
    kq.kq_embed(E, ids, 4, out)
    torch.cuda.synchronize()
    assert kq.kq_device_status(True) == kq.KQ_ERR_RANGE
    o = out.cpu().numpy().reshape(4, 64)
    assert not o[1].any() and not o[2].any() and o[0].any() and o[3].any()
    assert kq.kq_device_status(True) == kq.KQ_OK


# ----------------------------------------------------------------------------
# the fp16 chain (fp16 activation in, fp16 output)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,n,k,had", [("pq2_0", 10240, 5120, 128), ("pq2_0", 300, 5120, 1024),
                                         ("pq2_0", 64, 17408, 128), ("pq2_0", 33, 1152, 128),
                                         ("q8_0", 1024, 2560, 0), ("q8_0", 40, 9728, 0), ("scale4", 300, 4128, 0)])
def test_f16_chain_matches_oracle(kq, wl, fmt, n, k, had):
    """fp16 x -> (sign flip and) transform in fp32 -> fp16 -> product in fp32 ->
    fp16 y (the Bonsai page, section 4.4).  Bound per row: the fp32 bound, the
    oracle's slack for transformed values next to an fp16 rounding midpoint,
    and half an fp16 step of the output."""
    sid = synth.stream_id("test", 0, 470 + n % 97)
    sh, sd = (wl.build_signs(k, 3, synth.stream_id("test", 1, 471)) if had == 1024 else (None, None))
    W = wl.build_matrix(fmt, n, k, 9, sid, had_block=(1024 if had == 1024 else None), signs=sd)
    x16 = synth.fill_host("x", k, 9, synth.stream_id("test", 1, 472)).astype(np.float16)
    y16 = torch.empty(n, dtype=torch.float16, device="cuda")
    nb = kq.kq_gemv_workspace_bytes(W, 1)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    kq.kq_gemv_f16(W, torch.from_numpy(x16).cuda(), y16, ws)
    _sync_ok(kq)
    w = synth.fill_host("w", n * k, 9, sid).reshape(n, k)
    y_ref, absdot, slack, _ = oracle.f16_chain_reference(fmt, w, x16, had if had else 128, sh)
    got = y16.cpu().numpy().astype(np.float64)
    mag = np.abs(y_ref) + TOL * absdot + slack
    bound = TOL * absdot + slack + 0.5 * np.spacing(mag.astype(np.float16)).astype(np.float64) * (1 + 2.0**-10)
    err = np.abs(got - y_ref)
    assert np.all(err <= bound), float(np.max(err / np.maximum(bound, 1e-300)))
    if fmt != "pq2_0":  # no transform: the fp32 GEMV of the same input, rounded once
        y32 = _run_gemv(kq, W, torch.from_numpy(x16.astype(np.float32)).cuda())
        assert np.array_equal(got, y32.astype(np.float16).astype(np.float64))


# ----------------------------------------------------------------------------
# the page's rotation: n = 1024 blocks with a sign vector
# ----------------------------------------------------------------------------

def _page_reference(w, X, signs):
    """Oracle with R = H_1024 S / 32: W' = W R^T (rows rotated, then
    quantized) and x' = R x per activation row.  Returns (blocks, y, absdot)."""
    n, k = w.shape
    _, w_rot = oracle.rotate_rows(w, 1024, signs=signs)
    blocks = oracle.pq2_0_quantize(w_rot)
    deq = oracle.pq2_0_dequant(blocks, n, k)
    X = np.atleast_2d(X)
    y, a = oracle.gemm(deq, oracle.rotate_rows(X, 1024, signs=signs)[0])
    return blocks, y, a


def test_device_signed_rotation_bit_identical_to_host(kq, wl):
    for k, block in ((6144, 1024), (5120, 1024), (2048, 128)):
        sh, sd = wl.build_signs(k, 0, synth.stream_id("test", 1, 410 + block))
        x = np.random.default_rng(k).standard_normal((5, k)).astype(np.float32)
        out = torch.empty(5 * k, dtype=torch.float32, device="cuda")
        kq.kq_rotate_blockwise(torch.from_numpy(x).cuda(), out, 5, k, block, sd)
        _sync_ok(kq)
        assert np.array_equal(out.cpu().numpy().reshape(5, k), kq.kq_rotate_blockwise_host(x, block, sh))


@pytest.mark.parametrize("n,k", [(300, 5120), (64, 17408), (1000, 1024), (40, 6144)])
@pytest.mark.parametrize("with_signs", [True, False])
def test_pq2_0_page_rotation_matches_oracle(kq, consumer, wl, n, k, with_signs):
    """PQ2_0 with the page's n = 1024 rotation: device planes equal the
    oracle's bytes; the GEMV, the split GEMV, the streaming small-M path (the
    transform passes in the upper half of the staging buffer) and the
    tensor-core path are within the bound."""
    sid = synth.stream_id("test", 0, 420 + n)
    sh, sd = wl.build_signs(k, 1, synth.stream_id("test", 1, 421 + k)) if with_signs else (None, None)
    W = wl.build_matrix("pq2_0", n, k, 6, sid, had_block=1024, signs=sd)
    w = synth.fill_host("w", n * k, 6, sid).reshape(n, k)
    X = synth.fill_host("x", 16 * k, 6, synth.stream_id("test", 1, 422)).reshape(16, k)
    blocks, y_ref, absdot = _page_reference(w, X, sh)
    assert np.array_equal(_planes_as_blocks(kq, W), blocks)
    Xd = torch.from_numpy(X).cuda()
    y = _run_gemv(kq, W, Xd[0])
    ok, worst = oracle.within_bound(y, y_ref[0], absdot[0], TOL)
    assert ok, ("gemv", worst)
    y3 = _run_gemv(kq, W, Xd[0], splits=3)
    ok, worst = oracle.within_bound(y3, y_ref[0], absdot[0], TOL)
    assert ok, ("split 3", worst)
    for m in (3, 4, 16):
        Y = torch.empty(m * n, dtype=torch.float32, device="cuda")
        nb = kq.kq_gemv_workspace_bytes(W, m)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
        kq.kq_gemm_small_m(W, Xd[:m].reshape(-1), m, Y, ws)
        _sync_ok(kq)
        ok, worst = oracle.within_bound(Y.cpu().numpy().reshape(m, n), y_ref[:m], absdot[:m], TOL)
        assert ok, (m, worst)


def test_decode_plans_with_page_rotation(kq, consumer, wl):
    """Unlinked and linked plans over matrices of three K widths sharing one
    sign vector per width, as on the page."""
    widths = (5120, 6144, 17408)
    signs = {k: wl.build_signs(k, 2, synth.stream_id("test", 1, 430 + i)) for i, k in enumerate(widths)}
    spec = [(6144, 5120), (5120, 6144), (17408, 5120), (5120, 17408)]
    mats, host, rows = [], [], []
    rng = np.random.default_rng(8)
    for i, (n, k) in enumerate(spec):
        sid = synth.stream_id("test", 0, 440 + i)
        mats.append(wl.build_matrix("pq2_0", n, k, 7, sid, had_block=1024, signs=signs[k][1]))
        r = np.unique(np.r_[0, n - 1, rng.integers(0, n, size=30)])  # sampled rows: the oracle is O(n k 1024)
        rows.append(r)
        host.append(synth.matrix_rows_host(n, k, r, 7, sid))
    y_offsets = np.cumsum([0] + [n for n, _ in spec])
    # unlinked: every matrix its own packed input
    xs = [synth.fill_host("x", k, 7, synth.stream_id("test", 1, 450 + i)) for i, (_, k) in enumerate(spec)]
    plan = kq.DecodePlan(mats)
    y = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    plan.step(torch.from_numpy(np.concatenate(xs)).cuda(), y)
    _sync_ok(kq)
    yh = y.cpu().numpy()
    for i, (n, k) in enumerate(spec):
        _, y_ref, absdot = _page_reference(host[i], xs[i], signs[k][0])
        ok, worst = oracle.within_bound(yh[y_offsets[i] + rows[i]], y_ref[0], absdot[0], TOL)
        assert ok, ("unlinked", i, worst)
    plan.close()
    # linked: 0 -> 1 (prefix of 6144 outputs) -> 2 -> 3, a chain of four stages
    links = [(0, 0, 0, 1.0), (2, 1, 0, 0.5), (2, 2, 1, 0.25), (2, 3, 2, 0.125)]
    plan = kq.DecodePlan(mats, links)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    y = torch.full((plan.y_floats,), float("nan"), dtype=torch.float32, device="cuda")
    plan.step(torch.from_numpy(xs[0]).cuda(), y, ws)
    _sync_ok(kq)
    yh = y.cpu().numpy()
    xin = _linked_inputs(links, [k for _, k in spec], [xs[0]], yh, y_offsets)
    for i, (n, k) in enumerate(spec):
        _, y_ref, absdot = _page_reference(host[i], xin[i], signs[k][0])
        ok, worst = oracle.within_bound(yh[y_offsets[i] + rows[i]], y_ref[0], absdot[0], TOL)
        assert ok, ("linked", i, worst)
    plan.close()


def _linked_inputs(links, ks, x_packed, yh, y_offsets):
    """The activation every matrix of a linked plan reads: its packed slot,
    its group's input, or fp32(alpha * prefix of an earlier output) computed
    on the host from the device output."""
    xin, slot = [], 0
    for i, (src, _, of, alpha) in enumerate(links):
        if src == synth.SRC_PACKED:
            xin.append(x_packed[slot])
            slot += 1
        elif src == synth.SRC_INPUT_OF:
            xin.append(xin[of])
        else:
            o = int(y_offsets[of])
            xin.append((np.float32(alpha) * yh[o:o + ks[i]]).astype(np.float32))
    return xin


# (n, k) and link (src, stage, of, alpha) of a small chain: a grouped stage of
# three matrices (K split, ragged rows), a prefix of an output with a scale,
# a group reading an output, an empty stage, a second packed input, and a
# stage with enough row blocks to need no split
_CHAIN = [((200, 4096), (0, 0, 0, 1.0)), ((64, 4096), (1, 0, 0, 1.0)), ((300, 4096), (1, 0, 0, 1.0)),
          ((512, 256), (2, 1, 2, 0.5)), ((1000, 512), (2, 2, 3, 0.125)), ((333, 512), (1, 2, 4, 1.0)),
          ((256, 896), (2, 4, 4, 0.03125)), ((40, 256), (0, 4, 0, 1.0)), ((40000, 256), (2, 5, 6, 0.0625)),
          ((96, 128), (2, 6, 8, 3.0))]


@pytest.mark.parametrize("fmt", ["q8_0", "pq2_0", "scale4"])
def test_linked_plan_chain(kq, wl, fmt):
    mats, host, links = [], [], []
    for i, ((n, k), lk) in enumerate(_CHAIN):
        sw = synth.stream_id("test", 0, 360 + i)
        mats.append(wl.build_matrix(fmt, n, k, 5, sw))
        host.append(synth.fill_host("w", n * k, 5, sw).reshape(n, k))
        links.append(lk)
    plan = kq.DecodePlan(mats, links)
    assert plan.stages == 7 and plan.split_matrices > 0
    xp = [synth.fill_host("x", _CHAIN[i][0][1], 5, synth.stream_id("test", 1, 360 + i))
          for i, lk in enumerate(links) if lk[0] == synth.SRC_PACKED]
    x = torch.from_numpy(np.concatenate(xp)).cuda()
    assert plan.x_floats == x.numel()
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    y_offsets = np.cumsum([0] + [W.n for W in mats])
    outs = []
    for rep in range(2):
        # stale data must never be read: outputs and partials start as NaN
        y = torch.full((plan.y_floats,), float("nan"), dtype=torch.float32, device="cuda")
        ws.view(torch.float32).fill_(float("nan"))
        plan.step(x, y, ws)
        _sync_ok(kq)
        outs.append(y.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])  # deterministic
    yh = outs[0]
    assert np.isfinite(yh).all()
    xin = _linked_inputs(links, [W.k for W in mats], xp, yh, y_offsets)
    for i, (W, w) in enumerate(zip(mats, host)):
        _, _, y_ref, absdot = oracle.reference(fmt, w, xin[i])
        ok, worst = oracle.within_bound(yh[y_offsets[i]:y_offsets[i + 1]], y_ref, absdot, TOL)
        assert ok, (fmt, i, worst)
    plan.close()


def test_linked_plan_exact_integer_chain_tolerance_zero(kq):
    """A Q8_0 chain whose every product and partial sum is exact in fp32
    (power-of-two scales, small integer activations, |W| |x| below 2^24
    units of the result's granularity): the device outputs, including row
    blocks cut between CTAs and read back as sums of partials, must equal
    the oracle's FP64 values exactly.  Every block's scale is pinned to 2^-5
    by a code of 127 at its first position, where the activation is always
    zero (packed inputs are zero there, and rows r % 32 == 0 are zero rows,
    so every output read as a later activation is zero there too)."""
    rng = np.random.default_rng(21)
    # (n, k), (src, stage, of, alpha): a grouped stage of small matrices with
    # long K (its row blocks are cut many ways), prefixes of outputs, a
    # ragged K chunk (992) and scales alpha != 1
    spec = [((512, 2048), (0, 0, 0, 1.0)), ((384, 2048), (1, 0, 0, 1.0)), ((2048, 512), (2, 1, 0, 1.0)),
            ((1000, 2048), (2, 2, 2, 0.5)), ((256, 992), (2, 3, 3, 2.0))]
    mats, deqs, links = [], [], []
    for (n, k), lk in spec:
        q = rng.choice([-1, 0, 0, 0, 1], size=(n, k))
        q[:, ::32] = 127
        q[::32, :] = 0
        w = (q * 2.0**-5).astype(np.float32)
        blocks = oracle.q8_0_quantize(w)
        W = kq.QMatrix("q8_0", n, k)
        kq.kq_prepare(W, torch.from_numpy(blocks.reshape(-1)).cuda())
        mats.append(W)
        deqs.append(oracle.q8_0_dequant(blocks, n, k))
        links.append(lk)
    plan = kq.DecodePlan(mats, links)
    assert plan.split_matrices > 0
    x0 = rng.integers(-4, 5, size=2048).astype(np.float32)
    x0[::32] = 0.0
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ws.view(torch.float32).fill_(float("nan"))
    y = torch.full((plan.y_floats,), float("nan"), dtype=torch.float32, device="cuda")
    plan.step(torch.from_numpy(x0).cuda(), y, ws)
    _sync_ok(kq)
    yh = y.cpu().numpy()
    offs = np.cumsum([0] + [n for (n, _), _ in spec])
    xin, gran = [x0.astype(np.float64)], [1.0]  # activation values and their granularity
    for i, ((n, k), (src, _, of, alpha)) in enumerate(spec):
        if i > 0:
            if src == synth.SRC_INPUT_OF:
                xin.append(xin[of])
                gran.append(gran[of])
            else:
                xin.append(alpha * yh[offs[of]:offs[of] + k].astype(np.float64))
                gran.append(alpha * 2.0**-5 * gran[of])
        y_ref, absdot = oracle.gemv(deqs[i], xin[i])
        assert (absdot / (2.0**-5 * gran[i])).max() < 2.0**24  # every partial sum is exact
        assert np.array_equal(yh[offs[i]:offs[i + 1]].astype(np.float64), y_ref), i
    plan.close()


def test_linked_plan_cuts_row_blocks_only_where_it_pays(kq, wl):
    """The plan deals each stage to the SMs either in equal byte shares
    (cutting row blocks) or whole row blocks, whichever loads the busiest SM
    less.  Two 17408 x 5120 PQ2_0 matrices (136 row blocks of 5 chunks) go
    whole onto one SM each when there are at least 136 SMs; a 5120 x 6144
    stage (120 chunks) is cut when there are more SMs than chunks.  Sampled
    rows of each output match the oracle on the activation read."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    spec = [((17408, 5120), (0, 0, 0, 1.0)), ((17408, 5120), (1, 0, 0, 1.0)), ((5120, 6144), (2, 1, 0, 0.5))]
    seed = 7
    streams = [synth.stream_id("test", 0, 390 + i) for i in range(len(spec))]
    mats = [wl.build_matrix("pq2_0", n, k, seed, sw) for ((n, k), _), sw in zip(spec, streams)]
    plan = kq.DecodePlan(mats, [lk for _, lk in spec])
    if sms >= 136 and sms > 120:
        assert plan.split_matrices == 1  # only the 120-chunk stage is cut
    x0 = synth.fill_host("x", 5120, seed, synth.stream_id("test", 1, 390))
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ws.view(torch.float32).fill_(float("nan"))
    y = torch.full((plan.y_floats,), float("nan"), dtype=torch.float32, device="cuda")
    plan.step(torch.from_numpy(x0).cuda(), y, ws)
    _sync_ok(kq)
    yh = y.cpu().numpy()
    offs = np.cumsum([0] + [n for (n, _), _ in spec])
    xin = [x0, x0, (np.float32(0.5) * yh[: 6144]).astype(np.float32)]
    rng = np.random.default_rng(3)
    for i, ((n, k), _) in enumerate(spec):
        rows = np.unique(np.r_[0, n - 1, rng.integers(0, n, size=8)])
        w = synth.matrix_rows_host(n, k, rows, seed, streams[i])
        deq = oracle.pq2_0_dequant(oracle.pq2_0_quantize(oracle.rotate_rows(w)[1]), rows.size, k)
        y_ref, absdot = oracle.gemv(deq, oracle.rotate_rows(xin[i])[0])
        ok, worst = oracle.within_bound(yh[offs[i] + rows], y_ref, absdot, TOL)
        assert ok, (i, worst)
    plan.close()


@pytest.mark.parametrize("fmt", ["q8_0", "pq2_0"])
@pytest.mark.parametrize("linked,pinned", [(False, True), (True, True), (False, False), (True, False)])
def test_decode_step_host_matches_device_step(kq, consumer, wl, fmt, linked, pinned):
    """kq_decode_step_host (host buffers in and out) gives bitwise the outputs
    of kq_decode_step on the same inputs.  Pinned buffers: the kernel reads
    the activations through their device mapping (the device buffer d_x is
    left untouched) and a one-stage plan writes its outputs there; a plan
    with stages copies its outputs back.  Pageable buffers: both copies."""
    spec = [((300, 1024), (0, 0, 0, 1.0)), ((200, 1024), (1, 0, 0, 1.0)), ((64, 256), (2, 1, 0, 0.5))]
    if fmt == "pq2_0":
        spec[2] = ((64, 128), (2, 1, 0, 0.5))
    mats = [wl.build_matrix(fmt, n, k, 9, synth.stream_id("test", 0, 395 + i)) for i, ((n, k), _) in enumerate(spec)]
    plan = kq.DecodePlan(mats, [lk for _, lk in spec] if linked else None)
    xh = torch.from_numpy(synth.fill_host("x", plan.x_floats, 9, synth.stream_id("test", 1, 395)))
    yh = torch.full((plan.y_floats,), float("nan"), dtype=torch.float32)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    nb = plan.workspace_bytes
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
    dx = torch.full((plan.x_floats,), float("nan"), dtype=torch.float32, device="cuda")
    dy = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    plan.step_host(xh, yh, dx, dy, ws)
    torch.cuda.synchronize()
    _sync_ok(kq)
    assert torch.isnan(dx).all() == pinned  # read in place when pinned, copied in otherwise
    y2 = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    plan.step(xh.cuda(), y2, ws)
    _sync_ok(kq)
    assert torch.equal(yh, y2.cpu())
    plan.close()


def test_decode_step_host_misaligned_pinned_buffers_are_copied(kq, wl):
    """Page-locked host buffers whose device mapping is not 16-byte aligned
    are served by copies (the kernel's in-place path needs 16-byte rows):
    d_x is written, and the outputs still equal kq_decode_step's bit for bit."""
    mats = [wl.build_matrix("pq2_0", n, k, 9, synth.stream_id("test", 0, 398 + i))
            for i, (n, k) in enumerate([(300, 1024), (96, 512)])]
    plan = kq.DecodePlan(mats)
    xbig = torch.empty(plan.x_floats + 1, dtype=torch.float32).pin_memory()
    ybig = torch.full((plan.y_floats + 1,), float("nan"), dtype=torch.float32).pin_memory()
    xh, yh = xbig[1:], ybig[1:]  # 4 bytes past a 16-byte boundary
    xh.copy_(torch.from_numpy(synth.fill_host("x", plan.x_floats, 9, synth.stream_id("test", 1, 398))))
    dx = torch.full((plan.x_floats,), float("nan"), dtype=torch.float32, device="cuda")
    dy = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    plan.step_host(xh, yh, dx, dy, None)
    torch.cuda.synchronize()
    _sync_ok(kq)
    assert torch.equal(dx.cpu(), xh)  # copied in
    y2 = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    plan.step(xh.cuda(), y2, None)
    _sync_ok(kq)
    assert torch.equal(yh, y2.cpu())
    plan.close()


@pytest.mark.parametrize("seed", range(4))
def test_random_shapes_every_path_matches_oracle(kq, wl, seed):
    """Seeded random cases: format, ragged n, k a random number of blocks
    (ragged chunk tails), activation rows m and the entry point (GEMV, forced
    split-K, small-M routing, the tensor-core GEMM with forced splits), every
    row against the oracle."""
    rng = np.random.default_rng(7000 + seed)
    for case in range(6):
        fmt = str(rng.choice(["q8_0", "pq2_0", "scale4"]))
        block = 128 if fmt == "pq2_0" else 32
        n = int(rng.integers(1, 900))
        k = block * int(rng.integers(1, (48 if fmt == "pq2_0" else 160) + 1))
        path = str(rng.choice(["gemv", "splitk", "small_m", "tc"]))
        m = 1 if path == "gemv" else int(rng.choice([1, 2, 3, 4, 5, 16, 33, 64]))
        splits = int(rng.integers(0, 4))
        sw, sx = synth.stream_id("test", 0, 7100 + 10 * seed + case), synth.stream_id("test", 1, 7100 + 10 * seed + case)
        W = wl.build_matrix(fmt, n, k, 11, sw)
        X = wl.build_activation(k, 11, sx, rows=m)
        if path == "gemv":
            Y = _run_gemv(kq, W, X).reshape(1, n)
        elif path == "splitk":
            Y = _run_gemv(kq, W, X, splits=splits, m=m).reshape(m, n)
        elif path == "small_m":
            Yd = torch.empty(m * n, dtype=torch.float32, device="cuda")
            nb = kq.kq_gemv_workspace_bytes(W, m)
            ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
            kq.kq_gemm_small_m(W, X, m, Yd, ws)
            _sync_ok(kq)
            Y = Yd.cpu().numpy().reshape(m, n)
        else:
            Y = _run_tc(kq, W, X, m, splits)
        w = synth.fill_host("w", n * k, 11, sw).reshape(n, k)
        Xh = synth.fill_host("x", m * k, 11, sx).reshape(m, k)
        for i in range(m):
            _, _, y_ref, absdot = oracle.reference(fmt, w, Xh[i])
            ok, worst = oracle.within_bound(Y[i], y_ref, absdot, TOL)
            assert ok, (fmt, n, k, path, m, splits, i, worst)


def test_bounded_wait_timeout_is_reported_and_the_context_stays_usable(kq, wl):
    """A bounded device wait that runs out (an mbarrier phase that nothing
    completes, given up after ~1e6 cycles) is reported as KQ_ERR_TIMEOUT by
    kq_device_status, which then reads clean; the context keeps working: a
    GEMV afterwards matches the oracle."""
    assert kq.kq_device_status(True) == kq.KQ_OK
    kq.kq_selftest_bounded_wait(1_000_000)
    assert kq.kq_device_status(True) == kq.KQ_ERR_TIMEOUT
    assert kq.kq_device_status(True) == kq.KQ_OK  # cleared
    n, k = 300, 1024
    sw, sx = synth.stream_id("test", 0, 399), synth.stream_id("test", 1, 399)
    W = wl.build_matrix("pq2_0", n, k, 9, sw)
    x = wl.build_activation(k, 9, sx)
    y = _run_gemv(kq, W, x)
    _, _, y_ref, absdot = oracle.reference("pq2_0", synth.fill_host("w", n * k, 9, sw).reshape(n, k),
                                           synth.fill_host("x", k, 9, sx))
    ok, worst = oracle.within_bound(y, y_ref, absdot, TOL)
    assert ok, worst


def test_linked_plan_rejects_bad_links(kq, wl):
    mats = [wl.build_matrix("q8_0", 256, 256, 1, synth.stream_id("test", 0, 380 + i)) for i in range(3)]
    bad = [
        ([(0, 0, 0, 1.0), (1, 0, 0, 1.0), (2, 0, 1, 1.0)], kq.KQ_ERR_SHAPE),     # output read in its own stage
        ([(0, 1, 0, 1.0), (0, 0, 0, 1.0), (0, 2, 0, 1.0)], kq.KQ_ERR_SHAPE),     # decreasing stage
        ([(0, 0, 0, 1.0), (2, 1, 2, 1.0), (0, 2, 0, 1.0)], kq.KQ_ERR_INVALID_ARG),  # not an earlier matrix
        ([(0, 0, 0, 1.0), (3, 1, 0, 1.0), (0, 2, 0, 1.0)], kq.KQ_ERR_INVALID_ARG),  # unknown kind
        ([(0, 0, 0, 1.0), (2, 1, 0, float("inf")), (0, 2, 0, 1.0)], kq.KQ_ERR_INVALID_ARG),
    ]
    for links, status in bad:
        with pytest.raises(kq.KQError) as e:
            kq.DecodePlan(mats, links)
        assert e.value.status == status, links
    wide = wl.build_matrix("q8_0", 8, 512, 1, synth.stream_id("test", 0, 383))
    with pytest.raises(kq.KQError) as e:  # k = 512 exceeds the source's 256 outputs
        kq.DecodePlan([mats[0], wide], [(0, 0, 0, 1.0), (2, 1, 0, 1.0)])
    assert e.value.status == kq.KQ_ERR_SHAPE
    plan = kq.DecodePlan(mats, [(0, 0, 0, 1.0), (2, 1, 0, 1.0), (2, 2, 1, 1.0)])
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    y = torch.empty(plan.y_floats, dtype=torch.float32, device="cuda")
    with pytest.raises(kq.KQError) as e:
        plan.step(x, y, None)
    assert e.value.status == kq.KQ_ERR_WORKSPACE
    plan.close()


@pytest.mark.slow
@pytest.mark.parametrize("config", ["qwen3_4b_q8_0_step", "bonsai_27b_pq2_0_step"])
def test_linked_decode_step_full_size_sampled_rows(kq, wl, config):
    """The model-ordered chain of a whole decode step (stage by stage, one
    cooperative launch): sampled rows of every 5th projection and the head,
    each against the oracle on the activation it read."""
    W = wl.DecodeWorkload(config, seed=0, linked=True)
    W.y.fill_(float("nan"))
    W.step()
    _sync_ok(kq)
    y = W.y.cpu().numpy()
    assert np.isfinite(y).all()
    ks = [k for _, _, _, k in W.mats_spec]
    xp = [synth.fill_host("x", ks[i], W.seed, synth.stream_id(config, synth.ROLE_X, i)) for i in W.packed]
    xin = _linked_inputs(W.links, ks, xp, y, W.y_offsets)
    rng = np.random.default_rng(1)
    worst_all = 0.0
    for i, (_, fmt, n, k) in enumerate(W.mats_spec):
        if i % 5 and i != len(W.mats_spec) - 1:
            continue
        rows = np.unique(np.r_[0, n - 1, rng.integers(0, n, size=6)])
        w = synth.matrix_rows_host(n, k, rows, W.seed, synth.stream_id(config, synth.ROLE_W, i))
        if fmt == "pq2_0":
            deq = oracle.pq2_0_dequant(oracle.pq2_0_quantize(oracle.rotate_rows(w)[1]), rows.size, k)
            x64 = oracle.rotate_rows(xin[i])[0]
        else:
            deq = oracle.q8_0_dequant(oracle.q8_0_quantize(w), rows.size, k)
            x64 = xin[i].astype(np.float64)
        y_ref, absdot = oracle.gemv(deq, x64)
        ok, worst = oracle.within_bound(y[int(W.y_offsets[i]) + rows], y_ref, absdot, TOL)
        assert ok, (config, i, worst)
        worst_all = max(worst_all, worst)
    y2 = W.y.clone()
    W.step()
    _sync_ok(kq)
    assert torch.equal(W.y, y2)
    print(f"{config} linked: {W.plan.stages} stages, {W.plan.split_matrices} split, worst error/bound {worst_all:.3g}")
    W.close()


@pytest.mark.slow
@pytest.mark.parametrize("config", ["qwen3_4b_q8_0_step", "bonsai_27b_pq2_0_step"])
def test_decode_step_full_size_sampled_rows(kq, consumer, wl, config):
    W = wl.DecodeWorkload(config, seed=0)
    W.step()
    _sync_ok(kq)
    y = W.y.cpu().numpy()
    rng = np.random.default_rng(0)
    worst_all = 0.0
    for i, (_, fmt, n, k) in enumerate(W.mats_spec):
        if i % 7 and i != len(W.mats_spec) - 1:
            continue  # every 7th projection and the head
        rows = np.unique(np.r_[0, n - 1, rng.integers(0, n, size=6)])
        w, xh = W.host_rows(i, rows)
        if fmt == "pq2_0":
            blocks = oracle.pq2_0_quantize(oracle.rotate_rows(w)[1])
            deq = oracle.pq2_0_dequant(blocks, rows.size, k)
            x64 = oracle.rotate_rows(xh)[0]
        else:
            blocks = oracle.q8_0_quantize(w)
            deq = oracle.q8_0_dequant(blocks, rows.size, k)
            x64 = xh.astype(np.float64)
        # the device planes of these rows hold the oracle's bytes
        Wm = W.mats[i]
        nb = k // kq.kq_block_size(fmt)
        rb = kq.kq_codes_bytes(fmt, 1, k)
        ss = kq.kq_scale_stride(fmt, k)
        for t, r in enumerate(rows):
            codes = Wm.codes[int(r) * rb:(int(r) + 1) * rb].cpu().numpy()
            scales = Wm.scales[int(r) * ss:int(r) * ss + nb].cpu().numpy().view(np.uint16)
            assert np.array_equal(codes, blocks[t, :, 2:].reshape(-1))
            assert np.array_equal(scales, blocks[t, :, 0].astype(np.uint16) | (blocks[t, :, 1].astype(np.uint16) << 8))
        y_ref, absdot = oracle.gemv(deq, x64)
        off = int(W.y_offsets[i])
        ok, worst = oracle.within_bound(y[off + rows], y_ref, absdot, TOL)
        assert ok, (config, i, worst)
        worst_all = max(worst_all, worst)
    W.close()
    print(f"{config}: worst error/bound over sampled rows {worst_all:.3g}")
