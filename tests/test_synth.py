"""The seeded input generator against an independent Philox4x64-10 (numpy's
bit generator) and the published known-answer vector, plus the statistics
and grid properties the workloads rely on."""
import numpy as np
import pytest

import synth


def test_philox_known_answer_zero_counter_zero_key():
    # Random123 known-answer vector for philox4x64-10, counter 0 and key 0
    out = synth.philox_block([0, 0, 0, 0], [0, 0])
    assert [int(v) for v in out] == [0x16554D9ECA36314C, 0xDB20FE9D672D0FDC, 0xD7E772CEE186176B, 0x7E68B68AEC7BA23B]


@pytest.mark.parametrize("key", [(0, 0), (1, 2), (2**63 + 5, 123456789), (0xFFFFFFFFFFFFFFFF, 7)])
@pytest.mark.parametrize("ctr", [(0, 0, 0, 0), (41, 3, 0, 9), (2**64 - 2, 0, 0, 0)])
def test_philox_matches_numpy(key, ctr):
    # numpy's Philox advances the counter by one before each block
    bg = np.random.Philox(counter=np.array(ctr, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
    expect = bg.random_raw(4)
    c1 = list(ctr)
    c1[0] = (c1[0] + 1) % 2**64
    if c1[0] == 0:
        c1[1] += 1
    got = synth.philox_block(c1, key)
    assert np.array_equal(got, expect)


def test_weights_distribution_and_grid():
    w = synth.fill_host("w", 2_000_000, 0, synth.stream_id("test", 0, 100))
    assert abs(w.mean()) < 1e-4
    assert abs(w.std() - 0.02) < 1e-4
    m = w.astype(np.float64) * 2.0**20
    assert np.array_equal(m, np.round(m))
    assert np.abs(m).max() < 2**17  # so a 128-block sum stays below 2^24 quanta


def test_activation_distribution_and_grid():
    x = synth.fill_host("x", 2_000_000, 0, synth.stream_id("test", 1, 100))
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    m = x.astype(np.float64) * 2.0**16
    assert np.array_equal(m, np.round(m))


def test_fill_offsets_and_streams():
    s = synth.stream_id("test", 0, 101)
    full = synth.fill_host("w", 1000, 3, s)
    assert np.array_equal(synth.fill_host("w", 300, 3, s, first_index=500), full[500:800])
    assert not np.array_equal(synth.fill_host("w", 1000, 3, s + 1), full)
    assert not np.array_equal(synth.fill_host("w", 1000, 4, s), full)
    rows = synth.matrix_rows_host(10, 100, [7, 2], 3, s)
    assert np.array_equal(rows[0], full[700:800]) and np.array_equal(rows[1], full[200:300])
