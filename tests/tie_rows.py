"""Rows whose quantisation meets exact ties (TEST INPUTS, hand-worked codes).

Every row below is built so that each step before the rounding is exact in
fp32: the scale and zero point are powers of two or small multiples of them,
the row's own minimum and maximum produce exactly that scale, and every
element divided by the scale lands on k + 1/2.  The rounding rule is then the
only thing that decides a code, and the codes below were worked by hand with
ties going to the even neighbour (0.5 -> 0, 1.5 -> 2, 2.5 -> 2, -0.5 -> 0,
-1.5 -> -2, -2.5 -> -2).  Rounding half away from zero would give 1, 2, 3,
-1, -2, -3 instead, so a code path that used it fails.

Which rule applies: the write rounds codes half to even (vLLM PR #40835
review summary, 关键源码片段: `rounds_before_store=False`, the INT4 path rounds
by itself; the rule itself is the reading taken for the pages' "round").

Nothing here computes the method: the rows are inputs, the expected codes are
literals.
"""
import numpy as np

# --- INT4 / INT2 asymmetric per-token-head rows -----------------------------
# S = 0.25 and M = -1.5 (both exact binary16); the row holds M (t = 0) and
# M + levels * S (t = levels) so the row's own min / max give exactly S and M.
# t = (x - M) / S for each element; the code is rne(t) clamped to the range.
S_ASYM, M_ASYM = 0.25, -1.5
INT4_T = [0.0, 15.0, 0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, 7.5, 8.5, 9.5, 10.5, 11.5, 12.5, 13.5, 14.5]
INT4_CODES = [0, 15, 0, 2, 2, 4, 4, 6, 6, 8, 8, 10, 10, 12, 12, 14, 14]
INT2_T = [0.0, 3.0, 0.5, 1.5, 2.5, 0.5, 1.5, 2.5]
INT2_CODES = [0, 3, 0, 2, 2, 0, 2, 2]

# --- INT4 with the zero point in the scale ----------------------------------
# t = x / s_t with s_t = 0.125: the row spans t = -2.5 .. 12.5, so lo = -0.3125,
# hi = 1.5625, s = (hi - lo) / 15 = 0.125 exactly (bits 0x3E000000, low four
# bits already zero).  The zero point is rne(-lo / s_t) = rne(2.5) = 2 (half
# away would give 3); each code is clamp(rne(t) + 2, 0, 15).
S_STEGO = 0.125
STEGO_T = [-2.5, 12.5, -1.5, -0.5, 0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, 7.5, 8.5, 9.5, 10.5, 11.5]
STEGO_CODES = [0, 14, 0, 2, 2, 4, 4, 6, 6, 8, 8, 10, 10, 12, 12, 14]
STEGO_ZP = 2
STEGO_PAD = [0x02, 0x00, 0x00, 0x3E]

# --- INT8 per channel ---------------------------------------------------------
# Channel c has s_c = 2^(c % 7 - 3).  Token 0 is 127 s_c (the amax, so the
# scale amax / 127 is exactly s_c), token 1 is -127 s_c, then tokens at
# t = j + 1/2 for j = -127 .. 125 (t = -126.5 .. 125.5): codes are the even
# neighbour of t.
INT8_FIRST_CODES = [127, -127, -126, -126, -124, -124]     # t = 127, -127, -126.5, -125.5, -124.5, -123.5
INT8_LAST_CODES = [122, 124, 124, 126]                     # t = 122.5, 123.5, 124.5, 125.5


def int8_channel_scales(D):
    return 2.0 ** (np.arange(D) % 7 - 3)


def int8_channel_t():
    j = np.arange(-127, 126)
    return np.concatenate([[127.0, -127.0], j + 0.5])


def even_neighbour_of_half(t):
    """Reference rule spelled out on half-integers only: the integer of the
    pair {t - 1/2, t + 1/2} that is even.  Used to expand the pattern for the
    long INT8 channel list; the literal lists above were checked against it."""
    t = np.asarray(t, np.float64)
    lo = t - 0.5
    return np.where(np.mod(lo, 2) == 0, lo, lo + 1).astype(np.int64)


def _tile(pattern, D):
    return np.array([pattern[i % len(pattern)] for i in range(D)])


def asym_row(mode_bits, D):
    """(x [D] float32, codes [D]) for the INT4 (bits 4) or INT2 (bits 2) row."""
    t = _tile(INT4_T if mode_bits == 4 else INT2_T, D)
    codes = _tile(INT4_CODES if mode_bits == 4 else INT2_CODES, D)
    x = (M_ASYM + t * S_ASYM).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), M_ASYM + t * S_ASYM)
    return x, codes


def stego_row(D):
    t = _tile(STEGO_T, D)
    codes = _tile(STEGO_CODES, D)
    x = (t * S_STEGO).astype(np.float32)
    return x, codes


def int8_channel_tokens(D):
    """(x [T, D] float32, codes [T, D]) for one kv head."""
    s = int8_channel_scales(D)
    t = int8_channel_t()
    x = (t[:, None] * s[None, :]).astype(np.float32)
    codes = np.concatenate([[127, -127], even_neighbour_of_half(t[2:])])
    return x, np.repeat(codes[:, None], D, axis=1)


def pre_rotate(y, signs):
    """Input x whose forward rotation H (signs * x) is exactly y: x = signs *
    (H y) / D, with H the Sylvester Hadamard matrix.  Exact in fp32 for the
    short dyadic rows above (every partial sum is a small multiple of 2^-9)."""
    D = len(y)
    i = np.arange(D)
    pc = np.vectorize(lambda a: bin(a).count("1"))(i[:, None] & i[None, :])
    H = np.where(pc % 2 == 0, 1.0, -1.0)
    x = signs.astype(np.float64) * (H @ y.astype(np.float64)) / D
    x32 = x.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x)
    return x32
