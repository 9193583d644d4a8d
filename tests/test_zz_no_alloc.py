"""The allocation-free split-K entry point, through the C ABI.

It serves callers that cannot allocate device memory where they run the
product; its split-K partials live in a scratch array the library keeps in
device memory.  The test checks it against the regular entry point (which
takes a caller workspace) on two calls in a row, so that leftovers of the
first call cannot leak into the second, and that oversized plans are refused.
This file is collected last on purpose: it must also pass after every other
test has run in the same process."""
import ctypes

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
    return kq


def _regular(kq, W, X, m, splits):
    Y = torch.empty(m * W.n, dtype=torch.float32, device="cuda")
    nbytes = kq.kq_gemm_splitk_workspace_bytes(W, m, splits)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    kq.kq_gemm_splitk(W, X, m, Y, splits, ws)
    torch.cuda.synchronize()
    return Y.cpu().numpy()


def _noalloc(kq, W, X, m, splits):
    Y = torch.full((m * W.n,), float("nan"), dtype=torch.float32, device="cuda")
    lib = kq.lib()
    rc = lib.kq_gemm_splitk_noalloc(ctypes.byref(W.desc), X.data_ptr(), m, Y.data_ptr(), splits,
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == kq.KQ_OK, lib.kq_last_error().decode()
    torch.cuda.synchronize()
    assert kq.kq_device_status(True) == kq.KQ_OK
    return Y.cpu().numpy()


@pytest.mark.parametrize("fmt,n,k,m,splits", [("pq2_0", 640, 5120, 1, 4), ("q8_0", 1024, 2560, 2, 5),
                                                ("pq2_0", 300, 20480, 1, 0)])
def test_noalloc_matches_regular_entry_point_twice(kq, fmt, n, k, m, splits):
    import workloads

    sw = synth.stream_id("test", 0, 500)
    W = workloads.build_matrix(fmt, n, k, 6, sw)
    w = synth.fill_host("w", n * k, 6, sw).reshape(n, k)
    for call in range(2):  # two calls in a row, different activations
        sx = synth.stream_id("test", 1, 500 + call)
        X = workloads.build_activation(k, 6, sx, rows=m)
        y_reg = _regular(kq, W, X, m, splits)
        y_na = _noalloc(kq, W, X, m, splits)
        assert np.array_equal(y_na, y_reg)  # same split plan, same bits
        Xh = synth.fill_host("x", m * k, 6, sx).reshape(m, k)
        for i in range(m):
            _, _, y_ref, absdot = oracle.reference(fmt, w, Xh[i])
            ok, worst = oracle.within_bound(y_na.reshape(m, n)[i], y_ref, absdot, TOL)
            assert ok, (call, i, worst)


def test_noalloc_call_allocates_no_device_memory(kq):
    """After a first call (which may load the library's device code on this
    device), a call leaves the device's free memory (cudaMemGetInfo)
    unchanged: nothing is allocated, by the library or by anything it calls."""
    import workloads

    n, k, m, splits = 640, 5120, 1, 4
    W = workloads.build_matrix("pq2_0", n, k, 6, synth.stream_id("test", 0, 502))
    X = workloads.build_activation(k, 6, synth.stream_id("test", 1, 502))
    Y = torch.empty(m * n, dtype=torch.float32, device="cuda")
    lib = kq.lib()
    args = (ctypes.byref(W.desc), X.data_ptr(), m, Y.data_ptr(), splits, torch.cuda.current_stream().cuda_stream)
    assert lib.kq_gemm_splitk_noalloc(*args) == kq.KQ_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert lib.kq_gemm_splitk_noalloc(*args) == kq.KQ_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert kq.kq_device_status(True) == kq.KQ_OK


def test_noalloc_rejects_plans_beyond_its_scratch(kq):
    import workloads

    cap = kq.kq_gemm_splitk_noalloc_max_bytes()
    assert cap == 2 << 20
    n, k, splits = 16384, 9728, 38  # 38 splits x 16384 rows x 4 bytes > 2 MiB
    W = workloads.build_matrix("q8_0", n, k, 0, synth.stream_id("test", 0, 501))
    assert kq.kq_gemm_splitk_workspace_bytes(W, 1, splits) > cap
    X = workloads.build_activation(k, 0, synth.stream_id("test", 1, 501))
    Y = torch.full((n,), 3.0, device="cuda")
    with pytest.raises(kq.KQError) as e:
        kq.kq_gemm_splitk_noalloc(W, X, 1, Y, splits)
    assert e.value.status == kq.KQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(Y == 3.0)
