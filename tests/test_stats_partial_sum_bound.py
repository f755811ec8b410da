"""The bound stated for the bf16 elementwise statistics' sum: each thread of
the gate kernel adds its 256 fp16 scores into four float32 partial sums
(scores alternate between two packed pairs: word x of each 16-byte chunk goes
to pair x % 2, its low half to .x and its high half to .y), adds the four
partials in float32 and rounds the total times 2^32 once. The mean over a
thread's scores is then within 2^-18 of the exact mean. Checked against the
exact integer sum (every fp16 score times 2^24 is an integer) on scores with
widely spread exponents, where float32 additions round the most."""
import numpy as np


def _thread_sum_fixed(s16):
    # s16: 256 fp16 scores in the order one thread reads them (8 chunks x 4
    # 16-byte pieces x 4 words x 2 halves)
    acc = np.zeros((2, 2), np.float32)
    v = s16.astype(np.float32).reshape(8, 4, 4, 2)
    for k in range(8):
        for q in range(4):
            for x in range(4):
                for half in range(2):
                    acc[x % 2, half] = np.float32(acc[x % 2, half] + v[k, q, x, half])
    total = np.float32(np.float32(acc[0, 0] + acc[0, 1]) + np.float32(acc[1, 0] + acc[1, 1]))
    return int(np.rint(np.float64(total) * 2.0 ** 32))


def test_thread_mean_within_2_to_minus_18():
    rng = np.random.default_rng(7)
    worst = 0.0
    for trial in range(200):
        # exponents from 2^-24 to 1: the partials see every rounding step
        s = np.minimum(10.0 ** rng.uniform(-7.2, 0.0, 256), 1.0).astype(np.float16)
        if trial % 4 == 0:
            s[:] = np.float16(1.0) - np.float16(2.0 ** -11) * rng.integers(0, 8, 256).astype(np.float16)
        exact_2_24 = sum(int(round(float(x) * 2 ** 24)) for x in s.astype(np.float64))
        got = _thread_sum_fixed(s)
        err_mean = abs(got / 2.0 ** 32 - exact_2_24 / 2.0 ** 24) / 256
        worst = max(worst, err_mean)
    assert worst <= 2.0 ** -18


def test_exact_when_scores_share_a_binade():
    # scores in [0.25, 1): every partial stays exact, as on the headline's gates
    rng = np.random.default_rng(8)
    s = rng.uniform(0.25, 1.0, 256).astype(np.float16)
    exact_2_24 = sum(int(round(float(x) * 2 ** 24)) for x in s.astype(np.float64))
    assert _thread_sum_fixed(s) == exact_2_24 << 8
