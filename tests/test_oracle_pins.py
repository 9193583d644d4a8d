"""Pins of the FP64 oracle against things other than itself: library routines
(numpy float16, scipy's Hadamard), closed forms, hand-built blocks, figures
printed on the pages and brute force on tiny inputs."""
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page_figures():
    out = {}
    with open(os.path.join(GOLDEN, "page_figures.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                out[k] = float(v)
    return out


# ----------------------------------------------------------------------------
# binary16 conversion against numpy's IEEE float16 cast
# ----------------------------------------------------------------------------

def test_half_from_float_matches_numpy_on_many_values():
    rng = np.random.default_rng(1)
    # random bit patterns across the whole float32 range (finite only)
    bits = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # plus every float32 in a band around the binary16 range with dense exponents
    extra = np.concatenate([
        np.linspace(-70000, 70000, 200_001, dtype=np.float32),
        (rng.standard_normal(100_000) * 1e-5).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 2.0**-24, 2.0**-25, 3 * 2.0**-26,
                  2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11], dtype=np.float32),
    ])
    vals = np.concatenate([vals, extra])
    with np.errstate(over="ignore"):
        expect = vals.astype(np.float16).view(np.uint16)
    got = oracle.half_bits(vals)
    assert np.array_equal(got, expect)


def test_half_value_all_patterns_matches_numpy():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_value(pats)
    expect = pats.view(np.float16).astype(np.float32)
    nan = np.isnan(expect)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), expect[~nan].view(np.uint32))


# ----------------------------------------------------------------------------
# Hadamard
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024])
def test_hadamard_closed_forms(n):
    H = oracle.hadamard(n)
    assert np.array_equal(H @ H, n * np.eye(n))
    assert np.array_equal(H, H.T)
    assert np.array_equal(H, scipy.linalg.hadamard(n).astype(np.float64))


def test_hadamard_recursive_sylvester_construction():
    # independent construction: H_1 = [1], H_2n = [[H, H], [H, -H]]
    H = np.array([[1.0]])
    for _ in range(7):
        H = np.block([[H, H], [H, -H]])
    assert np.array_equal(oracle.hadamard(128), H)


def test_rotation_special_vectors():
    n = 128
    e0 = np.zeros(n, dtype=np.float32)
    e0[0] = 1
    r64, _ = oracle.rotate_rows(e0)
    assert np.allclose(r64, np.full(n, 1 / np.sqrt(n)), rtol=0, atol=1e-16)
    ones = np.ones(n, dtype=np.float32)
    r64, _ = oracle.rotate_rows(ones)
    expect = np.zeros(n)
    expect[0] = np.sqrt(n)
    assert np.allclose(r64, expect, rtol=0, atol=1e-13)


def test_rotation_is_orthogonal_involution():
    x = synth.fill_host("x", 3 * 128, 0, synth.stream_id("test", 1, 1)).reshape(3, 128)
    r64, r32 = oracle.rotate_rows(x)
    back64, _ = oracle.rotate_rows(r32)
    assert np.max(np.abs(back64 - x)) < 1e-5
    assert np.allclose(np.linalg.norm(r64, axis=1), np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-12)


def test_rotation_is_block_diagonal():
    k = 5 * 128
    x = synth.fill_host("x", k, 2, synth.stream_id("test", 1, 2))
    R = scipy.linalg.hadamard(128) / np.sqrt(128)
    B = scipy.linalg.block_diag(*([R] * 5))
    r64, _ = oracle.rotate_rows(x)
    assert np.max(np.abs(r64 - B @ x.astype(np.float64))) < 1e-12


def _signs(k, seed):
    return np.where(np.random.default_rng(seed).random(k) < 0.5, -1, 1).astype(np.int8)


def test_signed_rotation_all_plus_signs_is_the_unsigned_rotation():
    x = np.random.default_rng(3).standard_normal((3, 2048)).astype(np.float32)
    for n in (128, 1024):
        a64, a32 = oracle.rotate_rows(x, n)
        b64, b32 = oracle.rotate_rows(x, n, signs=np.ones(2048, dtype=np.int8))
        assert np.array_equal(a64, b64) and np.array_equal(a32, b32)


def test_signed_rotation_n1024_matches_scipy_hadamard():
    """The page's rotation (Bonsai page, sections 4.1-4.2): per 1024-block,
    x' = H_1024 (s * x) / 32 with scipy's Sylvester matrix, sign first; K =
    5120 is five blocks with one K-wide sign vector."""
    k = 5120
    s = _signs(k, 7)
    x = np.random.default_rng(4).standard_normal((2, k)).astype(np.float32)
    got64, got32 = oracle.rotate_rows(x, 1024, signs=s)
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    want = np.concatenate([(H @ (s[b * 1024:(b + 1) * 1024] * x[:, b * 1024:(b + 1) * 1024].astype(np.float64)).T).T
                           for b in range(5)], axis=1) / 32.0
    assert np.allclose(got64, want, rtol=0, atol=1e-12 * np.abs(x).sum())
    assert np.array_equal(got32, got64.astype(np.float32))
    # the transform is orthogonal: S H / 32 undoes it, and norms are kept
    back = np.concatenate([s[b * 1024:(b + 1) * 1024] * (H @ got64[:, b * 1024:(b + 1) * 1024].T).T / 32.0
                           for b in range(5)], axis=1)
    assert np.allclose(back, x, rtol=0, atol=1e-11)
    assert np.allclose(np.linalg.norm(got64, axis=1), np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-13)


def test_signed_rotation_of_a_signed_unit_vector():
    """R (s_j e_j) = H e_j / 32 (a column of H over 32): the sign cancels."""
    k = 2048
    s = _signs(k, 9)
    for j in (0, 5, 1023, 1024 + 77):
        x = np.zeros((1, k), dtype=np.float32)
        x[0, j] = float(s[j])
        got, _ = oracle.rotate_rows(x, 1024, signs=s)
        b, c = divmod(j, 1024)
        col = scipy.linalg.hadamard(1024)[:, c] / 32.0
        want = np.zeros(k)
        want[b * 1024:(b + 1) * 1024] = col
        assert np.array_equal(got[0], want)


def test_inverse_rotation_undoes_the_rotation_and_matches_scipy():
    """R^T R = I (orthogonality) through the two independent oracle routines,
    and the inverse against scipy's Hadamard matrix with the sign flip last."""
    k = 3072
    s = _signs(k, 21)
    x = np.random.default_rng(22).standard_normal((3, k)).astype(np.float32)
    for n, sg in ((128, None), (1024, s), (1024, None)):
        _, z32 = oracle.rotate_rows(x, n, signs=sg)
        back = oracle.rotate_rows_inverse(z32, n, signs=sg)
        assert np.max(np.abs(back - x)) <= 4e-6 * np.max(np.abs(x))  # z rounded to fp32 once
    z = np.random.default_rng(23).standard_normal((2, k)).astype(np.float32)
    H = scipy.linalg.hadamard(1024).astype(np.float64)
    want = np.concatenate([s[b * 1024:(b + 1) * 1024] * (H @ z[:, b * 1024:(b + 1) * 1024].astype(np.float64).T).T
                           for b in range(3)], axis=1) / 32.0
    assert np.allclose(oracle.rotate_rows_inverse(z, 1024, signs=s), want, rtol=0, atol=1e-12 * np.abs(z).sum())


def test_signed_rotation_rejects_bad_signs():
    x = np.zeros((1, 1024), dtype=np.float32)
    bad = np.ones(1024, dtype=np.int8)
    bad[3] = 0
    with pytest.raises(oracle.OracleError):
        oracle.rotate_rows(x, 1024, signs=bad)


def test_rotation_of_grid_weights_is_one_multiply_of_an_exact_sum():
    # Synthetic weights are integers times 2^-20, so H w is an exact integer
    # sum; the oracle must return fl64(fl64(1/sqrt(128)) * (H w)).
    w = synth.fill_host("w", 4 * 256, 3, synth.stream_id("test", 0, 3)).reshape(4, 256)
    m = np.round(w.astype(np.float64) * 2.0**20).astype(np.int64)
    assert np.array_equal(m.astype(np.float64) * 2.0**-20, w.astype(np.float64))
    H = scipy.linalg.hadamard(128).astype(np.int64)
    s = np.concatenate([m[:, :128] @ H.T, m[:, 128:] @ H.T], axis=1)  # exact integer H w
    expect64 = (1.0 / np.sqrt(128.0)) * (s.astype(np.float64) * 2.0**-20)
    r64, r32 = oracle.rotate_rows(w)
    assert np.array_equal(r64, expect64)
    assert np.array_equal(r32, expect64.astype(np.float32))


# ----------------------------------------------------------------------------
# Q8_0
# ----------------------------------------------------------------------------

def test_q8_0_block_size_from_page():
    fig = _page_figures()
    n_blocks = 128 // 32
    assert n_blocks * oracle.BLOCK_BYTES == fig["q8_0_bytes_per_128dim_row"]
    blocks = oracle.q8_0_quantize(np.zeros((1, 128), dtype=np.float32))
    assert blocks.nbytes == fig["q8_0_bytes_per_128dim_row"]


def test_q8_0_hand_built_block_round_trips_exactly():
    q = np.array([127, -127, 0, 1, -1, 5, -64, 100] + list(range(-50, 46, 4)), dtype=np.int64)
    assert q.size == 32
    w = (q * 2.0**-7).astype(np.float32)[None, :]
    blocks = oracle.q8_0_quantize(w)
    assert blocks.shape == (1, 1, 34)
    b = blocks[0, 0]
    # d = amax/127 = 2^-7 exactly -> fp16 0x2000, stored little endian first
    assert (b[0], b[1]) == (0x00, 0x20)
    assert np.array_equal(b[2:].view(np.int8).astype(np.int64), q)
    deq = oracle.q8_0_dequant(blocks, 1, 32)
    assert np.array_equal(deq, w)


def test_q8_0_rounds_half_away_from_zero():
    # amax = 127 * 2^-7 so d = 2^-7; values at exact halves of d
    vals = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5]
    w = np.zeros(32, dtype=np.float32)
    w[: len(vals)] = np.array(vals) * 2.0**-7
    q = oracle.q8_0_quantize(w[None])[0, 0, 2:].view(np.int8)
    assert list(q[: len(vals)]) == [127, 3, -3, 1, -1, 2, -2, 127, -127]


def test_q8_0_quantizes_against_the_fp16_rounded_scale():
    # amax = 1: d = 1/127 in fp32 is not a binary16 value; fp16(d) is a bit
    # smaller, so a weight at 100.497 d lands above the half way point of d_f.
    d = np.float32(1.0) / np.float32(127.0)
    d_f = np.float16(d).astype(np.float32)
    assert d_f != d
    w_val = np.float32(100.497) * d
    assert np.round(float(w_val) / float(d)) == 100
    assert np.round(float(w_val) / float(d_f)) == 101
    w = np.zeros(32, dtype=np.float32)
    w[0] = 1.0
    w[1] = w_val
    b = oracle.q8_0_quantize(w[None])[0, 0]
    assert int(b[2:].view(np.int8)[1]) == 101
    assert (int(b[0]) | (int(b[1]) << 8)) == int(np.float16(d).view(np.uint16))


def test_q8_0_zero_block_and_no_minus_128():
    w = np.zeros((2, 64), dtype=np.float32)
    w[1] = synth.fill_host("w", 64, 0, synth.stream_id("test", 0, 4))
    blocks = oracle.q8_0_quantize(w)
    assert not blocks[0].any()
    rng = np.random.default_rng(0)
    big = (rng.standard_normal((64, 512)) * rng.uniform(1e-3, 10, size=(64, 1))).astype(np.float32)
    codes = oracle.q8_0_quantize(big)[:, :, 2:].view(np.int8)
    assert codes.min() >= -127 and codes.max() <= 127
    # the largest magnitude of each block maps to +-127
    assert np.all(np.abs(codes).max(axis=2) == 127)


def test_q8_0_errors():
    with pytest.raises(oracle.OracleError):
        oracle.q8_0_quantize(np.zeros((1, 48), dtype=np.float32))
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 3] = np.nan
    with pytest.raises(oracle.OracleError):
        oracle.q8_0_quantize(w)
    w[0, 3] = 1e7  # amax/127 > 65504 does not fit the fp16 scale
    with pytest.raises(oracle.OracleError):
        oracle.q8_0_quantize(w)


def test_q8_0_dequant_error_bounded_by_half_step():
    w = synth.fill_host("w", 8 * 2560, 0, synth.stream_id("test", 0, 5)).reshape(8, 2560)
    blocks = oracle.q8_0_quantize(w)
    deq = oracle.q8_0_dequant(blocks, 8, 2560)
    d = oracle.half_value(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    step = np.repeat(d, 32, axis=1)
    assert np.all(np.abs(deq - w) <= 0.5 * step * (1 + 1e-6) + 1e-12)


# ----------------------------------------------------------------------------
# PQ2_0
# ----------------------------------------------------------------------------

def test_pq2_0_block_size_from_page():
    fig = _page_figures()
    blocks = oracle.pq2_0_quantize(np.ones((1, 128), dtype=np.float32))
    assert blocks.shape == (1, 1, fig["pq2_0_block_bytes"])
    assert blocks.nbytes * 8 / 128 == fig["pq2_0_bits_per_weight"]


def test_pq2_0_byte_layout_from_worked_examples():
    cases = []
    with open(os.path.join(GOLDEN, "pq2_0_bytes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                lhs, rhs = line.split("=")
                cases.append(([int(c) for c in lhs.split()], int(rhs, 16)))
    codes = []
    for c, _ in cases:
        codes += c
    codes += [1] * (128 - len(codes))
    w = (np.array(codes, dtype=np.float64) - 1) * 2.0**-4  # ternary grid, d = 2^-4
    b = oracle.pq2_0_quantize(w.astype(np.float32)[None])[0, 0]
    assert (int(b[0]) | (int(b[1]) << 8)) == 0x2C00  # fp16(2^-4)
    for i, (_, byte) in enumerate(cases):
        assert int(b[2 + i]) == byte
    assert np.all(b[2 + len(cases):] == 0x55)
    deq = oracle.pq2_0_dequant(b[None, None], 1, 128)[0]
    assert np.array_equal(deq, w.astype(np.float32))


def test_pq2_0_word_view():
    # Bonsai page, section 3.1 "Word view": bytes qs[4i..4i+3] read as a little
    # endian uint32 hold element 16i + j at bits 2j.
    w = synth.fill_host("w", 4 * 512, 1, synth.stream_id("test", 0, 6)).reshape(4, 512)
    _, w_rot = oracle.rotate_rows(w)
    blocks = oracle.pq2_0_quantize(w_rot)
    deq = oracle.pq2_0_dequant(blocks, 4, 512)
    d = oracle.half_value(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    words = np.ascontiguousarray(blocks[:, :, 2:]).view("<u4")  # [4, 4 blocks, 8 words]
    for r in range(4):
        for blk in range(4):
            for i in range(8):
                for j in range(16):
                    code = (int(words[r, blk, i]) >> (2 * j)) & 3
                    assert code in (0, 1, 2)
                    assert deq[r, blk * 128 + 16 * i + j] == np.float32(code - 1) * d[r, blk]


def test_pq2_0_scale_is_block_max_and_codes_ternary():
    w = synth.fill_host("w", 16 * 1024, 2, synth.stream_id("test", 0, 7)).reshape(16, 1024)
    _, w_rot = oracle.rotate_rows(w)
    blocks = oracle.pq2_0_quantize(w_rot)
    d = oracle.half_value(blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8))
    amax = np.abs(w_rot.reshape(16, 8, 128)).max(axis=2)
    assert np.array_equal(d, amax.astype(np.float16).astype(np.float32))
    codes = np.stack([(blocks[:, :, 2:] >> s) & 3 for s in (0, 2, 4, 6)], axis=-1)
    assert codes.max() <= 2  # code 3 never occurs
    # ternary round: |w'/d| < 1/2 -> 0 (code 1); else sign (half away from zero)
    deq = oracle.pq2_0_dequant(blocks, 16, 1024).reshape(16, 8, 128)
    ratio = w_rot.reshape(16, 8, 128).astype(np.float64) / d[:, :, None]
    expect = np.where(np.abs(ratio) >= 0.5, np.sign(ratio), 0.0) * d[:, :, None]
    assert np.array_equal(deq, expect.astype(np.float32))


def test_pq2_0_ties_and_zero_block():
    w = np.zeros((2, 128), dtype=np.float32)
    w[0, 0] = 1.0
    w[0, 1] = 0.5
    w[0, 2] = -0.5
    w[0, 3] = 0.49999997
    b = oracle.pq2_0_quantize(w)
    assert int(b[0, 0, 2]) == (2 | (2 << 2) | (0 << 4) | (1 << 6))
    assert np.all(b[1, 0, 2:] == 0x55) and b[1, 0, 0] == 0 and b[1, 0, 1] == 0


def test_ternary_all_ones_block_dots_to_zero_and_all_twos_to_d_sum():
    x = synth.fill_host("x", 128, 5, synth.stream_id("test", 1, 8))
    d_bits = 0x2E66  # an arbitrary fp16 scale
    blk = np.zeros((2, 1, 34), dtype=np.uint8)
    blk[:, 0, 0] = d_bits & 0xFF
    blk[:, 0, 1] = d_bits >> 8
    blk[0, 0, 2:] = 0x55  # every code 1 -> value 0
    blk[1, 0, 2:] = 0xAA  # every code 2 -> value +d
    deq = oracle.pq2_0_dequant(blk, 2, 128)
    x64, _ = oracle.rotate_rows(x)
    y, _ = oracle.gemv(deq, x64)
    assert y[0] == 0.0
    d = float(np.uint16(d_bits).view(np.float16))
    assert abs(y[1] - d * x64.sum()) <= 1e-12 * np.abs(x64).sum()


# ----------------------------------------------------------------------------
# GEMV
# ----------------------------------------------------------------------------

def _ptq1_0_golden():
    bytes_, blocks = [], []
    for line in open(os.path.join(GOLDEN, "ptq1_0_bytes.txt")):
        line = line.split("#")[0].strip()
        if line.startswith("byte "):
            lhs, rhs = line[5:].split("=")
            bytes_.append(([int(t) for t in lhs.split()], int(rhs)))
        elif line.startswith("block "):
            head, rest = line[6:].split(":")
            e, sgn = head.split()
            diffs = dict((int(a), int(b)) for a, b in (kv.split("=") for kv in rest.split()))
            blocks.append((int(e), int(sgn), diffs))
    return bytes_, blocks


def test_ptq1_0_byte_rule_from_page_worked_values():
    bytes_, _ = _ptq1_0_golden()
    assert len(bytes_) >= 7
    for trits, q in bytes_:
        assert oracle.ptq1_0_encode_byte(trits) == q, trits


def test_ptq1_0_trit_rule_inverts_the_byte_rule_for_every_byte():
    """Brute force over all 243 five-trit bytes (and the 81 four-trit qh
    bytes): the page's trit extraction returns every trit the byte rule
    packed."""
    import itertools

    for trits in itertools.product(range(3), repeat=5):
        q = oracle.ptq1_0_encode_byte(list(trits))
        assert 0 <= q <= 255
        assert [oracle.ptq1_0_decode_trit(q, n) for n in range(5)] == list(trits)


def test_ptq1_0_single_element_blocks_match_hand_worked_bytes():
    """The element-order table and the scale's place (last) on hand-built
    blocks."""
    _, blocks = _ptq1_0_golden()
    assert len(blocks) >= 5
    for e, sgn, diffs in blocks:
        w = np.zeros((1, 128), dtype=np.float32)
        w[0, e] = sgn * 2.0 ** -4
        got = oracle.ptq1_0_quantize(w)[0, 0]
        want = np.array([128] * 24 + [127, 127, 0x00, 0x2C], dtype=np.uint8)
        for b, v in diffs.items():
            want[b] = v
        assert np.array_equal(got, want), (e, got)
        deq = oracle.ptq1_0_dequant(got[None, None], 1, 128)
        assert np.array_equal(deq, w)


def test_ptq1_0_is_a_lossless_transcode_of_pq2_0():
    """Same trits and scale as PQ2_0 (the page: the two packs are lossless
    transcodes of each other): the dequantized matrices are equal."""
    w = synth.fill_host("w", 64 * 1024, 3, synth.stream_id("test", 0, 205)).reshape(64, 1024)
    _, w_rot = oracle.rotate_rows(w)
    a = oracle.ptq1_0_dequant(oracle.ptq1_0_quantize(w_rot), 64, 1024)
    b = oracle.pq2_0_dequant(oracle.pq2_0_quantize(w_rot), 64, 1024)
    assert np.array_equal(a, b)
    assert oracle.ptq1_0_quantize(w_rot).nbytes * 34 == oracle.pq2_0_quantize(w_rot).nbytes * 28


def _scale4_golden():
    cases = []
    for line in open(os.path.join(GOLDEN, "scale4_bytes.txt")):
        if line.startswith("#") or "|" not in line:
            continue
        head, hx = line.split("|")
        name, spec = head.split(":", 1)
        w = np.zeros(32, dtype=np.float32)
        for kv in spec.split()[1:]:
            j, v = kv.split(":")
            w[int(j)] = float(v) * 2.0 ** -7
        cases.append((name.strip(), w, bytes.fromhex(hx.strip())))
    return cases


def test_scale4_hand_worked_blocks():
    cases = _scale4_golden()
    assert len(cases) == 5
    for name, w, want in cases:
        got = oracle.scale4_quantize(w[None])[0, 0]
        assert bytes(got) == want, (name, bytes(got).hex())


def test_scale4_round_trip_of_grid_weights_is_exact():
    """w = d (q - 8) with d = -2^-7 and the extreme q = 0 present: the
    quantizer recovers every q and the dequantized block equals w."""
    rng = np.random.default_rng(12)
    for _ in range(20):
        q = rng.integers(1, 16, size=32)
        q[rng.integers(0, 32)] = 0
        w = ((q - 8) * -(2.0 ** -7)).astype(np.float32)[None]
        blocks = oracle.scale4_quantize(w)
        assert np.array_equal(oracle.scale4_dequant(blocks, 1, 32), w)


def test_scale4_dequant_error_bound_and_range():
    w = synth.fill_host("w", 16 * 1024, 4, synth.stream_id("test", 0, 206)).reshape(16, 1024)
    blocks = oracle.scale4_quantize(w)
    deq = oracle.scale4_dequant(blocks, 16, 1024)
    bits = blocks.reshape(-1, 18)[:, 0].astype(np.uint16) | (blocks.reshape(-1, 18)[:, 1].astype(np.uint16) << 8)
    d = np.abs(oracle.half_value(bits)).repeat(32)
    err = np.abs(deq.reshape(-1) - w.reshape(-1))
    # half a step, or one step for the one clamped value (q - 8 = +8 -> +7)
    assert np.all(err <= d * (1 + 2 ** -10) + 1e-12)
    assert np.mean(err <= d / 2 * (1 + 2 ** -10)) > 0.99
    with pytest.raises(oracle.OracleError):
        oracle.scale4_quantize(np.full((1, 32), 6e5, dtype=np.float32))  # |d| = 6e5/8 overflows fp16
    with pytest.raises(oracle.OracleError):
        oracle.scale4_quantize(np.zeros((1, 48), dtype=np.float32))


def test_gemv_brute_force_4x128_scale4():
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((4, 128)) * 0.02).astype(np.float32)
    x = rng.standard_normal(128).astype(np.float32)
    _, deq, y, a = oracle.scale4_reference(w, x)
    for i in range(4):
        want = sum(float(deq[i, j]) * float(x[j]) for j in range(128))
        assert abs(y[i] - want) <= 1e-12 * sum(abs(float(deq[i, j]) * float(x[j])) for j in range(128))
        assert abs(a[i] - sum(abs(float(deq[i, j]) * float(x[j])) for j in range(128))) <= 1e-12 * a[i]


def test_f16_chain_of_a_scaled_unit_vector():
    """x = c e_j in fp16: R x = (c / sqrt(128)) H[:, j] exactly, so x'16 is
    fp16(+-c / sqrt(128)) everywhere in the block, worked by hand: for
    c = 3, 3 / sqrt(128) = 0.26516504... -> fp16 0.2651367 (0x343E)."""
    w = np.zeros((2, 256), dtype=np.float32)
    w[0, :128] = 0.5  # some block scale; the y check below only needs x'
    x16 = np.zeros(256, dtype=np.float16)
    x16[5] = 3.0
    _, _, slack, xp16 = oracle.f16_chain_reference("pq2_0", w, x16)
    h = scipy.linalg.hadamard(128)[:, 5]
    want = np.float16(0.2651367)
    assert want.view(np.uint16) == 0x343E
    assert np.array_equal(xp16[:128], (h * want).astype(np.float16))
    assert not xp16[128:].any()
    assert np.all(slack == 0)


def test_f16_chain_exact_integer_case():
    """Q8_0 with integer codes, power-of-two scales and small integer fp16
    activations: the FP64 y is an exact integer multiple of 2^-5 that fp16
    holds exactly, so the chain's fp16 output equals it."""
    rng = np.random.default_rng(15)
    q = rng.integers(-127, 128, size=(6, 256))
    q[:, ::32] = 127
    w = (q * 2.0 ** -5).astype(np.float32)
    x16 = np.zeros(256, dtype=np.float16)  # eight nonzero activations: |y 2^5| <= 8 * 127 * 2 < 2^11
    x16[rng.choice(256, size=8, replace=False)] = rng.choice([-2, -1, 1, 2], size=8)
    y, _, slack, _ = oracle.f16_chain_reference("q8_0", w, x16)
    assert np.array_equal(y, (q @ x16.astype(np.int64)) * 2.0 ** -5)
    assert np.array_equal(y.astype(np.float16).astype(np.float64), y)  # 11 significant bits suffice
    assert not slack.any()


def _midpoint_case(x2):
    """The page's n = 1024 rotation (no signs) divides by 32 exactly, so
    R x is rational and can be placed on an fp16 rounding midpoint by hand.
    x = (1024, 1/2, x2, 0, ...) in fp16: R x_j = (1024 + s1 / 2 + s2 x2) / 32
    with s1 = (-1)^bit0(j), s2 = (-1)^bit1(j).  For even j that is
    32 + 2^-6 +- x2 / 32: within x2 / 32 of the midpoint 32 + 2^-6 between the
    fp16 values 32 and 32 + 2^-5 (fp16 step 2^-5 at 32, 2^-6 below it); for
    odd j it is 32 - 2^-6 +- x2 / 32, next to the fp16 value 32 - 2^-6 and
    half a step from any midpoint.  The weights are W = T R with T ternary
    (+-1/8, 0): R R = I with exact FP64 arithmetic on these values, so the
    rotated weights are T exactly and so is the dequantized matrix."""
    n, k = 6, 1024
    rng = np.random.default_rng(21)
    t = rng.integers(-1, 2, size=(n, k)) * 0.125
    t[:, ::128] = 0.125  # every 128-block has a nonzero weight: its scale is 1/8
    w = (t @ scipy.linalg.hadamard(k) / 32.0).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), t @ scipy.linalg.hadamard(k) / 32.0)  # exact in fp32
    x16 = np.zeros(k, dtype=np.float16)
    x16[:3] = [1024.0, 0.5, x2]
    assert float(x16[2]) == x2
    y, absdot, slack, xp16 = oracle.f16_chain_reference("pq2_0", w, x16, had=1024)
    return t, x16, y, absdot, slack, xp16


@pytest.mark.parametrize("x2", [2.0 ** -14, 2.0 ** -11])
def test_f16_chain_slack_at_an_fp16_midpoint(x2):
    """R x lies x2 / 32 (2^-19 or 2^-16) from an fp16 midpoint at every even
    j; the fp32 transform's error bound there is (log2 1024 + 3) 2^-24
    sum|x| / 32 = 13 * 2^-24 * (1024.5 + x2) / 32, about 2.48e-5, so both
    cases count as near.  Worked by hand: x'16_j is the exact value rounded
    once (32 + 2^-5 when bit1(j) = 0, above the midpoint; 32 when bit1 = 1,
    below it; 32 - 2^-6 for odd j); the fp16 step at a near position is
    max(c - lo, hi - c) = 2^-5 (c = 32: neighbours 32 - 2^-6 and 32 + 2^-5;
    c = 32 + 2^-5: 32 and 32 + 2^-4); so slack_i = 2^-5 sum_{j even} |T_ij|."""
    t, x16, y, absdot, slack, xp16 = _midpoint_case(x2)
    j = np.arange(1024)
    b0, b1 = j & 1, (j >> 1) & 1
    want16 = np.where(b0 == 0, np.where(b1 == 0, 32.0 + 2.0 ** -5, 32.0), 32.0 - 2.0 ** -6)
    assert np.array_equal(xp16.astype(np.float64), want16)
    want_slack = 2.0 ** -5 * np.abs(t[:, b0 == 0]).sum(axis=1)
    assert np.array_equal(slack, want_slack)
    assert np.array_equal(y, t @ want16)  # every term is a multiple of 2^-9: exact
    assert np.array_equal(absdot, np.abs(t) @ want16)


def test_f16_chain_no_slack_just_outside_the_bound():
    """x2 = 2^-10: R x is 2^-15 = 3.05e-5 from the midpoint, just above the
    error bound 13 * 2^-24 * (1024.5 + 2^-10) / 32 = 2.48e-5, so no position
    counts as near and the slack is zero; x'16 is the same correctly rounded
    transform."""
    _, _, _, _, slack, xp16 = _midpoint_case(2.0 ** -10)
    assert not slack.any()
    j = np.arange(1024)
    want16 = np.where(j & 1 == 0, np.where((j >> 1) & 1 == 0, 32.0 + 2.0 ** -5, 32.0), 32.0 - 2.0 ** -6)
    assert np.array_equal(xp16.astype(np.float64), want16)


def test_gemv_brute_force_4x128_pq2_0():
    w = synth.fill_host("w", 4 * 128, 9, synth.stream_id("test", 0, 9)).reshape(4, 128)
    x = synth.fill_host("x", 128, 9, synth.stream_id("test", 1, 9))
    blocks, deq, y, absdot = oracle.pq2_0_reference(w, x)
    # brute force along another route: (W' R) x with scipy's Hadamard,
    # products and sums by plain Python floats
    R = scipy.linalg.hadamard(128) / np.sqrt(128)
    for i in range(4):
        row = [sum(float(deq[i, c]) * float(R[c, j]) for c in range(128)) for j in range(128)]
        yi = sum(row[j] * float(x[j]) for j in range(128))
        assert abs(yi - y[i]) <= 1e-12 * max(1.0, absdot[i])
        assert absdot[i] >= abs(y[i])


def test_gemv_brute_force_4x128_q8_0():
    w = synth.fill_host("w", 4 * 128, 10, synth.stream_id("test", 0, 10)).reshape(4, 128)
    x = synth.fill_host("x", 128, 10, synth.stream_id("test", 1, 10))
    blocks, deq, y, absdot = oracle.q8_0_reference(w, x)
    for i in range(4):
        codes = blocks[i, :, 2:].view(np.int8).astype(int)
        scales = oracle.half_value(blocks[i, :, 0].astype(np.uint16) | (blocks[i, :, 1].astype(np.uint16) << 8))
        yi = 0.0
        ai = 0.0
        for b in range(4):
            for j in range(32):
                p = float(scales[b]) * int(codes[b, j]) * float(x[32 * b + j])
                yi += p
                ai += abs(p)
        assert abs(yi - y[i]) <= 1e-12 * max(1.0, ai)
        assert abs(ai - absdot[i]) <= 1e-12 * ai


def test_gemv_exact_integer_case():
    # integer codes, power-of-two scales, small integer activations: every
    # product and partial sum is an exact integer multiple of the scale, so the
    # FP64 sum must equal Python's integer arithmetic.
    rng = np.random.default_rng(7)
    n, k = 72, 128 * 3
    codes = rng.integers(-127, 128, size=(n, k))
    codes[:, ::32] = 127  # every block's max is 127 so d = 2^-5 exactly
    w = (codes * 2.0**-5).astype(np.float32)
    x = rng.integers(-8, 9, size=k).astype(np.float32)
    blocks, deq, y, absdot = oracle.q8_0_reference(w, x)
    assert np.array_equal(deq, w)
    exact = (codes @ x.astype(np.int64)) * 2.0**-5
    assert np.array_equal(y, exact)
    assert np.array_equal(absdot, (np.abs(codes) @ np.abs(x).astype(np.int64)) * 2.0**-5)


def test_gemv_row_subset_matches_full():
    w = synth.fill_host("w", 64 * 256, 11, synth.stream_id("test", 0, 11)).reshape(64, 256)
    x = synth.fill_host("x", 256, 11, synth.stream_id("test", 1, 11)).astype(np.float64)
    y, a = oracle.gemv(w, x)
    rows = np.array([63, 0, 17, 17, 40])
    ys, as_ = oracle.gemv(w, x, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(as_, a[rows])
    ys2, _ = oracle.gemv(w[rows], x, rows=rows, rows_are_packed=True, n_total=64)
    assert np.array_equal(ys2, y[rows])


def test_nonzero_mean_activation_case():
    # a DC offset in x must not hide errors behind cancellation: the bound is
    # taken on |w||x|, which grows with the offset while |y| may not.
    w = synth.fill_host("w", 8 * 512, 12, synth.stream_id("test", 0, 12)).reshape(8, 512)
    x = synth.fill_host("x", 512, 12, synth.stream_id("test", 1, 12)) + np.float32(3.0)
    _, _, y, absdot = oracle.pq2_0_reference(w, x)
    assert np.all(absdot > np.abs(y))


def test_within_bound_helper():
    ok, worst = oracle.within_bound([1.0, 2.0], np.array([1.0, 2.0005]), np.array([1.0, 10.0]))
    assert ok and worst == pytest.approx(0.5)
    ok, _ = oracle.within_bound([1.0], np.array([1.01]), np.array([1.0]))
    assert not ok


# ----------------------------------------------------------------------------
# Figures printed on the pages, against the workload shapes
# ----------------------------------------------------------------------------

def test_bonsai_shapes_match_page_figures():
    fig = _page_figures()
    mats = synth.bonsai_27b_projections()
    assert len(mats) == fig["folded_matrices"]
    for _, fmt, n, k in mats:
        assert fmt == "pq2_0"
        assert k % fig["kernel_constraint_k_multiple"] == 0
        assert n % fig["kernel_constraint_n_multiple"] == 0
    packed = sum(n * k // 128 * 34 for _, _, n, k in mats)
    assert abs(packed / 1e9 - fig["per_token_weight_traffic_gb"]) < 0.05
    head = fig["vocab_rows"] * fig["embedding_length"]
    assert round(head / 128 * 34 / 1e9, 2) == fig["vocab_table_packed_gb"]
    assert round(head * 2 / 1e9, 2) == fig["vocab_table_fp16_gb"]


def test_qwen3_4b_shapes():
    mats = synth.qwen3_4b_projections()
    assert len(mats) == 253
    assert sum(n * k for _, _, n, k in mats) == 4_022_272_000
    assert sum(n * k // 32 * 34 for _, _, n, k in mats) == 4_273_664_000
