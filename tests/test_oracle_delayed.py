"""Pins the oracle's delayed-scaling state against closed forms.

Closed form of the rule (newest amax at hist[0], update = max over the
window then roll): the multiplier used at step t+1 is
fmax / max(a_{t-H+1}, ..., a_t), where a_j is the amax seen at step j, as
long as that maximum is positive; before any positive amax it stays 1.
"""
import numpy as np
import pytest

import oracle as o


def _run(amaxes, H, fmt, algo=o.ALGO_MAX):
    st = o.state_init(H)
    used = []
    for a in amaxes:
        used.append(float(st[H]))
        x = np.float32([a, -a / 2, a / 4])
        o.quantize_delayed(x, fmt, st)
        o.update_scale(st, fmt, algo)
    return st, used


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
@pytest.mark.parametrize("H", [1, 4, 16])
def test_window_max_closed_form(fmt, H):
    rng = np.random.default_rng(H + 10 * fmt)
    amaxes = list(np.float32(rng.uniform(0.5, 4.0, 40)))
    amaxes[7] = np.float32(100.0)                    # spike
    amaxes[20] = np.float32(0.01)                    # dip
    st, used = _run(amaxes, H, fmt)
    fm = np.float32(o.fmax(fmt))
    assert used[0] == 1.0
    for t in range(1, len(amaxes)):
        win = max(amaxes[max(0, t - H):t])
        assert used[t] == fm / np.float32(win), t
    # history after the last update: [0, a_T, a_{T-1}, ...]
    T = len(amaxes)
    exp_hist = [0.0] + [float(amaxes[T - 1 - i]) for i in range(H - 1)]
    assert st[:H].tolist() == exp_hist
    assert st[H + 1] == np.float32(max(amaxes[T - H:])) / fm


def test_most_recent_algo():
    amaxes = [np.float32(v) for v in [2.0, 8.0, 1.0, 4.0]]
    st, used = _run(amaxes, 16, o.E4M3, o.ALGO_MOST_RECENT)
    assert used[1:] == [448.0 / 2.0, 448.0 / 8.0, 448.0 / 1.0]
    assert st[16] == np.float32(448.0) / np.float32(4.0)


def test_zero_and_nonfinite_amax_keep_the_scale():
    st = o.state_init(4)
    o.quantize_delayed(np.float32([2.0]), o.E4M3, st)
    o.update_scale(st, o.E4M3)
    m = st[4]
    for _ in range(4):                           # zeros push the 2.0 out of the window
        o.quantize_delayed(np.zeros(3, np.float32), o.E4M3, st)
        o.update_scale(st, o.E4M3)
    assert st[4] == m                            # window max 0 -> kept
    o.quantize_delayed(np.float32([np.inf]), o.E4M3, st)
    o.update_scale(st, o.E4M3)
    assert st[4] == m                            # window max inf -> kept


def test_stale_scale_is_used_for_the_current_cast():
    st = o.state_init(16)
    q, sat = o.quantize_delayed(np.float32([1000.0, 1.0]), o.E4M3, st)
    assert sat == 1 and q[0] == 0x7E and o.decode(o.E4M3, int(q[1])) == 1.0   # m = 1 at init
    assert st[0] == 1000.0


def test_two_tensors_sharing_a_role_combine_by_max():
    st = o.state_init(16)
    o.quantize_delayed(np.float32([3.0]), o.E5M2, st)
    o.quantize_delayed(np.float32([-7.0]), o.E5M2, st)
    assert st[0] == 7.0


def test_checkpoint_resume_is_bit_identical():
    rng = np.random.default_rng(11)
    xs = [rng.standard_normal(64).astype(np.float32) * (1 + t) for t in range(12)]
    st = o.state_init(16)
    for x in xs:
        o.quantize_delayed(x, o.E4M3, st)
        o.update_scale(st, o.E4M3)
    st2 = o.state_init(16)
    for x in xs[:5]:
        o.quantize_delayed(x, o.E4M3, st2)
        o.update_scale(st2, o.E4M3)
    saved = st2.copy()
    st3 = saved.copy()
    for x in xs[5:]:
        o.quantize_delayed(x, o.E4M3, st3)
        o.update_scale(st3, o.E4M3)
    assert st3.tobytes() == st.tobytes()
