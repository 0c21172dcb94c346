"""Compressor inputs whose RMSNorm sum of squares depends on the order of the
double additions (test input construction; numbers only, no kernel or oracle
arithmetic).

Two large channels y0, y1 in the first 64-channel group, every other channel
a small power of two.  Their squares sum to d times the midpoint between two
adjacent fp32 values.  Added in ascending channel order, every small square
is less than half an ulp of the running sum and is lost, so the mean square
rounds (ties to even) to one neighbour.  In the butterfly-then-groups order
the small squares meet each other first, survive, and push the mean square
to the other neighbour.

The pooled vector is produced exactly by a ratio-4 compressor at its first
boundary (position 3): the window is tokens 0..3 of the second block, all
scores are 0 (equal softmax weights, exp(0) = 1), so y = (kv_0 + kv_1 +
kv_2 + kv_3) / 4.  A 16-bit integer n times 2^e is kv_0 + kv_1 with both bf16
(its high and low 8 bits), so y0 and y1 are exact.  A ratio-128 stream gets
the same vector at position 127 from 128 tokens (token_rows_c128).
"""
import numpy as np

# found by a seeded search over 16-bit pairs (d, n0, n1, exponent, small)
CASES = {
    128: (48008, 38056, -15, 2.0 ** -27),
    512: (39688, 37528, -15, 2.0 ** -27),
    576: (50580, 33216, -15, 2.0 ** -27),
}


def butterfly_sum(y):
    """Sum of squares in the association the compressor fixes."""
    ss = 0.0
    for g in range(y.size // 64):
        v = [float(y[64 * g + 2 * l]) ** 2 + float(y[64 * g + 2 * l + 1]) ** 2 for l in range(32)]
        for dist in (16, 8, 4, 2, 1):
            v = [v[l] + v[l ^ dist] for l in range(32)]
        ss += v[0]
    return ss


def ascending_sum(y):
    ss = 0.0
    for c in range(y.size):
        ss += float(y[c]) * float(y[c])
    return ss


def pooled_vector(d):
    n0, n1, e, small = CASES[d]
    y = np.full(d, small, np.float32)
    y[0] = np.float32(n0 * 2.0 ** e)
    y[1] = np.float32(n1 * 2.0 ** e)
    return y


def bf16_bits_exact(x):
    """bf16 bit patterns of float32 values that bf16 holds exactly."""
    u = np.asarray(x, np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def token_rows(d):
    """kv_score rows (bf16 bits) of tokens 0..3 for a ratio-4 stream of dim d:
    [kv block a | kv block b | score block a | score block b]."""
    n0, n1, e, small = CASES[d]
    kv = np.zeros((4, d), np.float32)
    for c, n in ((0, n0), (1, n1)):
        kv[0, c] = np.float32((n & 0xFF00) * 2.0 ** e * 4)
        kv[1, c] = np.float32((n & 0x00FF) * 2.0 ** e * 4)
    kv[0, 2:] = np.float32(4 * small)
    rows = np.zeros((4, 4 * d), np.uint16)
    rows[:, d:2 * d] = bf16_bits_exact(kv)
    return rows


def token_rows_c128(d):
    """kv_score rows (bf16 bits) of tokens 0..127 for a ratio-128 stream of dim
    d, [kv | score]: at its first boundary (position 127) the window is all
    128 tokens with scores 0, so y = (sum of kv) / 128 with the same two-row
    split of n0, n1 as the ratio-4 rows (every sum exact)."""
    n0, n1, e, small = CASES[d]
    kv = np.zeros((128, d), np.float32)
    for c, n in ((0, n0), (1, n1)):
        kv[0, c] = np.float32((n & 0xFF00) * 2.0 ** e * 128)
        kv[1, c] = np.float32((n & 0x00FF) * 2.0 ** e * 128)
    kv[0, 2:] = np.float32(128 * small)
    rows = np.zeros((128, 2 * d), np.uint16)
    rows[:, :d] = bf16_bits_exact(kv)
    return rows


def mean_square_pair(d):
    """(ascending-order, butterfly-order) mean squares rounded to fp32."""
    y = pooled_vector(d)
    return np.float32(ascending_sum(y) / d), np.float32(butterfly_sum(y) / d)
