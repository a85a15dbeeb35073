"""Pins the CPU oracle to the numbers the pages print (tests/golden).

Each case cites its page and section in the fixture.  A plausible slip in the
oracle -- ties away from zero instead of to even, a division where the page
multiplies, a wrong maximum -- changes at least one of these numbers.
"""
import numpy as np
import pytest

import oracle as o


def test_int8_absmax_vector(golden):
    inp, exp, _ = golden["int8_absmax_vector"]
    q, step = o.int8_absmax(inp)
    assert q.tolist() == [int(v) for v in exp]
    _, deq, _ = golden["int8_absmax_dequant"]
    assert np.round(q.astype(np.float64) * float(step), 3).tolist() == deq
    _, st, _ = golden["int8_absmax_step"]
    assert round(float(step), 4) == st[0]


def test_int8_absmax_outlier(golden):
    inp, exp, _ = golden["int8_absmax_outlier"]
    q, step = o.int8_absmax(inp)
    assert q.tolist() == [int(v) for v in exp]
    _, st, _ = golden["int8_outlier_step"]
    assert round(float(step), 3) == st[0]
    # "all numbers up to 0.5 in absolute value got 5 levels (from -2 to 2)"
    small = np.linspace(-0.5, 0.5, 1001, dtype=np.float32)
    qs, _ = o.int8_absmax(np.concatenate([small, np.float32([30.0])]))
    assert sorted(set(qs[:-1].tolist())) == [-2, -1, 0, 1, 2]


def test_int8_absmax_block_of_two(golden):
    inp, exp, _ = golden["int8_block2_first"]
    q, _ = o.int8_absmax(inp)
    assert q.tolist() == [int(v) for v in exp]


def test_fp8_maxima(golden):
    assert o.fmax(o.E4M3) == golden["e4m3_max"][1][0]
    assert o.fmax(o.E5M2) == golden["e5m2_max"][1][0]


def test_e4m3_spacing_and_64_plus_3(golden):
    (a, b), (gap,), _ = golden["e4m3_spacing_64_128"]
    assert o.decode(o.E4M3, o.encode(o.E4M3, a)) == a
    assert o.decode(o.E4M3, o.encode(o.E4M3, b)) == b
    assert b - a == gap
    # no E4M3 value strictly between 64 and 72
    vals = sorted({o.decode(o.E4M3, c) for c in range(0x7F)})
    assert not [v for v in vals if a < v < b]
    (x, y), (r,), _ = golden["e4m3_64_plus_3"]
    assert o.decode(o.E4M3, o.encode(o.E4M3, x + y)) == r


def test_e4m3_running_sum_stalls(golden):
    (term, n, promote), (final,), _ = golden["e4m3_sum_100_threes"]
    total, stall = o.fp8_running_sum(o.E4M3, term, int(n), int(promote))
    assert total == final
    _, (step,), _ = golden["e4m3_sum_stall_step"]
    assert stall == step


def test_e4m3_promotion_every_8_pins_ties_to_even(golden):
    (term, n, promote), (final,), _ = golden["e4m3_sum_promote_8"]
    total, _ = o.fp8_running_sum(o.E4M3, term, int(n), int(promote))
    assert total == final
    # The 8-term partial under ties-to-even is 24 (21 -> 20, 23 -> 24);
    # ties away from zero would give 26 and a total of 324.
    part, _ = o.fp8_running_sum(o.E4M3, term, 8, 0)
    assert part == 24.0


def test_bf16_257(golden):
    (v,), (r,), _ = golden["bf16_257"]
    bits = o.bf16_from_f32(v)
    assert float(o.bf16_bits_to_f32(np.array([bits], dtype=np.uint16))[0]) == r
    (a, b), (gap,), _ = golden["bf16_spacing_256"]
    assert o.bf16_from_f32(a) + 1 == o.bf16_from_f32(b)
    assert b - a == gap


def test_delayed_worked_example(golden):
    """Transformer Scaling, worked example: amax 240 in the history gives the
    multiplier 448/240 ~ 1.87; 120 maps to 224; a spike of 300 maps to ~560
    and clips at 448.  Run as two steps of the delayed state."""
    (hist_amax,), (scale,), _ = golden["delayed_scale"]
    st = o.state_init(16)
    q, _ = o.quantize_delayed(np.float32([hist_amax, -hist_amax]), o.E4M3, st)  # step 1 sees amax 240
    o.update_scale(st, o.E4M3)
    m = st[16]
    assert round(float(m), 2) == scale
    (_, v120), (r120,), _ = golden["delayed_maps_120"]
    (_, v300), (r300,), _ = golden["delayed_spike_300"]
    q, sat = o.quantize_delayed(np.float32([v120, v300]), o.E4M3, st)      # step 2 uses the stale scale
    assert o.decode(o.E4M3, int(q[0])) == r120
    assert o.decode(o.E4M3, int(q[1])) == r300
    assert sat == 1
    _, (pre,), _ = golden["delayed_spike_scaled"]
    assert abs(float(np.float32(v300) * m) - pre) / pre < 0.01
    # the spike enters the history: the next step's scale covers it
    o.update_scale(st, o.E4M3)
    assert st[16] == np.float32(448.0) / np.float32(300.0)


def test_history_length_of_recipe(golden):
    H = int(golden["te_history_len"][1][0])
    st = o.state_init(H)
    o.quantize_delayed(np.float32([100.0]), o.E4M3, st)
    o.update_scale(st, o.E4M3)
    for _ in range(H - 1):          # the 100 stays in the window for H updates
        o.quantize_delayed(np.float32([1.0]), o.E4M3, st)
        o.update_scale(st, o.E4M3)
        assert st[H] == np.float32(448.0) / np.float32(100.0)
    o.quantize_delayed(np.float32([1.0]), o.E4M3, st)
    o.update_scale(st, o.E4M3)
    assert st[H] == np.float32(448.0)
