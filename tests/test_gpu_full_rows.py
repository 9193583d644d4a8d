"""Full-size decode steps checked on every row against the oracle.

* Qwen3-4B-shaped Q8_0 step: all 253 projections, every row, in the
  unlinked plan and in the model-ordered linked plan over the same device
  matrices.
* Bonsai-27B-shaped PQ2_0 step: every row of one projection of each of its
  seven (n, k) shapes (the last one in model order, deepest in the chain)
  and of the 248320-row output head, in the unlinked plan under both
  one-row consumers and in the linked plan.

The host regenerates every weight row from its seeded stream, quantizes it in
the oracle (rotating first for PQ2_0), checks that the device planes hold the
oracle's bytes, and multiplies in FP64, in row chunks spread over the host's
cores; one oracle pass serves every device result of a projection.  A linked
projection is checked on the activation it read (its packed input, or fp32
alpha times the prefix of an earlier device output)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

import oracle  # noqa: E402
import synth  # noqa: E402

TOL = 1e-4
CHUNK_WEIGHTS = 1 << 21  # weights per host task


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


def _sync_ok(kq):
    torch.cuda.synchronize()
    assert kq.kq_device_status(True) == kq.KQ_OK


def _linked_inputs(links, ks, x_packed, yh, y_offsets):
    """Per matrix of a linked plan, the activation it reads (fp32)."""
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


def _rows_task(fmt, n, k, seed, stream, r0, r1, x64s, codes, scales):
    """Oracle blocks, plane check and FP64 products of rows r0..r1-1."""
    oracle.set_threads(1)  # this pool thread's own setting: the chunks run in parallel instead
    w = synth.fill_host("w", (r1 - r0) * k, seed, stream, r0 * k).reshape(r1 - r0, k)
    if fmt == "pq2_0":
        blocks = oracle.pq2_0_quantize(oracle.rotate_rows(w)[1])
        deq = oracle.pq2_0_dequant(blocks, r1 - r0, k)
    else:
        blocks = oracle.q8_0_quantize(w)
        deq = oracle.q8_0_dequant(blocks, r1 - r0, k)
    nb = blocks.shape[1]
    planes_ok = (np.array_equal(codes[r0:r1], blocks[:, :, 2:].reshape(r1 - r0, -1))
                 and np.array_equal(scales[r0:r1, :nb],
                                    blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8)))
    return r0, r1, planes_ok, [oracle.gemv(deq, x) for x in x64s]


def _check_projection(kq, pool, config, seed, i, spec, Wm, x_list, y_list, tag):
    """Every row of projection i: x_list[j] is the fp32 activation that device
    output y_list[j] (this projection's slice) was computed from.  Returns the
    worst |error| / bound over the rows and outputs."""
    _, fmt, n, k = spec
    codes = Wm.codes.cpu().numpy()[: n * kq.kq_codes_bytes(fmt, 1, k)].reshape(n, -1)
    ss = kq.kq_scale_stride(fmt, k)
    scales = Wm.scales.cpu().numpy().view(np.uint16)[: n * ss].reshape(n, ss)
    uniq = []  # distinct activations (a linked group shares its input)
    which = []
    for x in x_list:
        for u, xu in enumerate(uniq):
            if xu is x or np.array_equal(xu, x):
                which.append(u)
                break
        else:
            which.append(len(uniq))
            uniq.append(x)
    x64s = [oracle.rotate_rows(x)[0] if fmt == "pq2_0" else x.astype(np.float64) for x in uniq]
    stream = synth.stream_id(config, synth.ROLE_W, i)
    step = max(1, CHUNK_WEIGHTS // k)
    futs = [pool.submit(_rows_task, fmt, n, k, seed, stream, r0, min(n, r0 + step), x64s, codes, scales)
            for r0 in range(0, n, step)]
    worst = 0.0
    for f in futs:
        r0, r1, planes_ok, prods = f.result()
        assert planes_ok, (tag, i, r0, r1, "device planes differ from the oracle's blocks")
        for j, y in enumerate(y_list):
            y_ref, absdot = prods[which[j]]
            ok, wv = oracle.within_bound(y[r0:r1], y_ref, absdot, TOL)
            assert ok, (tag, i, j, r0, wv)
            worst = max(worst, wv)
    return worst


def _linked_step(kq, W, config):
    """The linked (model-ordered) plan over the workload's device matrices:
    returns (links, host output)."""
    links = synth.decode_links(config)
    plan = kq.DecodePlan(W.mats, links)
    k0 = W.mats_spec[0][3]
    assert plan.x_floats == k0
    xl = W.x[:k0]  # the first projection's input is the chain's only packed input
    yl = torch.full((plan.y_floats,), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device="cuda")
    plan.step(xl, yl, ws)
    _sync_ok(kq)
    out = yl.cpu().numpy()
    plan.close()
    assert np.isfinite(out).all()
    return links, out


def _unlinked_step(kq, W):
    W.y.fill_(float("nan"))
    W.step()
    _sync_ok(kq)
    out = W.y.cpu().numpy()
    assert np.isfinite(out).all()
    return out


def _run(kq, config, pick, consumers):
    import workloads

    seed = 0
    W = workloads.DecodeWorkload(config, seed=seed)
    outs = []
    for c in consumers:
        kq.kq_set_pq2_0_consumer(c)
        outs.append(_unlinked_step(kq, W))
    kq.kq_set_pq2_0_consumer(kq.KQ_PQ2_0_MMA_SYNC)
    links, yl = _linked_step(kq, W, config)
    ks = [k for _, _, _, k in W.mats_spec]
    xu = [synth.fill_host("x", ks[i], seed, synth.stream_id(config, synth.ROLE_X, i)) for i in range(len(ks))]
    xin = _linked_inputs(links, ks, [xu[0]], yl, W.y_offsets)
    worst = 0.0
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as pool:
        for i in pick:
            o0, o1 = int(W.y_offsets[i]), int(W.y_offsets[i + 1])
            ys = [y[o0:o1] for y in outs] + [yl[o0:o1]]
            xs = [xu[i]] * len(outs) + [xin[i]]
            worst = max(worst, _check_projection(kq, pool, config, seed, i, W.mats_spec[i], W.mats[i], xs, ys,
                                                 config))
    W.close()
    return worst


def test_qwen3_4b_q8_0_step_every_row(kq):
    config = "qwen3_4b_q8_0_step"
    n_mats = len(synth.workload(config))
    assert n_mats == 253
    worst = _run(kq, config, range(n_mats), [kq.KQ_PQ2_0_MMA_SYNC])
    print(f"{config}: 253 projections, every row, unlinked and linked: worst error/bound {worst:.3g}")


def test_bonsai_27b_pq2_0_step_every_row_of_each_shape_and_the_head(kq):
    config = "bonsai_27b_pq2_0_step"
    spec = synth.workload(config)
    last = {}
    for i, (_, _, n, k) in enumerate(spec):
        last[(n, k)] = i
    pick = sorted(last.values())
    assert len(pick) == 8 and spec[pick[-1]][2] == 248320  # seven layer shapes, then the head
    worst = _run(kq, config, pick, [kq.KQ_PQ2_0_MMA_SYNC, kq.KQ_PQ2_0_TCGEN05])
    print(f"{config}: every row of {[spec[i][0] for i in pick]}, both consumers and linked: "
          f"worst error/bound {worst:.3g}")
