"""Pins of the CPU oracle to facts fixed outside itself.

Each test checks the oracle against something it does not share code with:
values the pages print (tests/golden/page_constants.txt), closed forms
(Sylvester's Hadamard matrix, worked grid rows), a library routine (numpy's
IEEE binary16 conversion), or brute force (numpy softmax attention on inputs
whose quantisation is exact).  A plausible slip in the oracle -- a dropped
sign flip, a wrong butterfly stride, a swapped nibble, a scale off by one
level, a window off by one, a sentinel that leaks -- fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import kvq_inputs as gen
import tie_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INT4, INT2, INT8 = oracle.MODE_INT4, oracle.MODE_INT2, oracle.MODE_INT8
STEGO = oracle.MODE_INT4_STEGO
I8T, F8T = oracle.MODE_INT8_TOKEN_HEAD, oracle.MODE_FP8_TOKEN_HEAD


def page_constants():
    out = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            k, v = [s.strip() for s in line.split("=")]
            out[k] = float(v)
    return out


def sylvester(n):
    i = np.arange(n)
    pc = np.vectorize(lambda a: bin(a).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def f16_of_pad(row, data_bytes):
    s = np.frombuffer(row[data_bytes:data_bytes + 2].tobytes(), dtype=np.float16)[0]
    m = np.frombuffer(row[data_bytes + 2:data_bytes + 4].tobytes(), dtype=np.float16)[0]
    return float(s), float(m)


def test_rounding_mode_nearest():
    assert oracle.lib().orc_rounding_mode_is_nearest() == 1


# --------------------------------------------------------------------------
# constants printed on the pages

def test_page_constants_ranges_and_rows():
    c = page_constants()
    # offset encoding: stored nibble u -> signed q = u - 8 spans the page's range
    assert oracle.signed_code(INT4, 0) == c["int4_quant_min"]
    assert oracle.signed_code(INT4, 15) == c["int4_quant_max"]
    assert [oracle.signed_code(INT2, u) for u in range(4)] == [-2, -1, 0, 1]
    assert oracle.row_bytes(INT4, 128) == c["int4_row_bytes_head_dim_128"]
    assert oracle.row_bytes(INT4, 64) == c["int4_row_bytes_head_dim_64"]
    assert oracle.row_bytes(INT4, 128) == 128 * c["int4_data_bytes_per_head_dim"] + c["scale_pad_bytes"]
    # INT2 packs twice as densely with the same pad; INT8 is one byte per element
    assert oracle.row_bytes(INT2, 128) == 128 // 4 + c["scale_pad_bytes"]
    assert oracle.row_bytes(INT8, 128) == 128 * c["storage_bytes_per_element_of_cache"]
    assert oracle.row_bytes(INT4, 96) == 0  # unsupported head_dim


# --------------------------------------------------------------------------
# IEEE binary16 against numpy's conversion (a library routine)

def test_f16_decode_all_patterns_match_numpy():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_decode(int(p)) for p in pats[::7]], dtype=np.float32)
    r = ref[::7]
    fin = np.isfinite(r)
    assert np.array_equal(got[fin], r[fin])
    assert np.array_equal(np.isinf(got), np.isinf(r))


def test_f16_round_matches_numpy_incl_ties_and_subnormals():
    rng = np.random.default_rng(1)
    vals = [0.0, -0.0, 1.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0 ** -24, 2.0 ** -25,
            3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
            1024.5, 1025.5, 2049.0, 2051.0, -7.00048828125]
    vals += list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-9, 5, 3000))
    for x in vals:
        xf = np.float32(x)
        with np.errstate(over="ignore"):
            want = np.array([xf]).astype(np.float16).view(np.uint16)[0]
        assert oracle.f16_round(float(xf)) == int(want), x


def test_f16_saturate():
    assert oracle.f16_saturate(1e9) == 0x7BFF
    assert oracle.f16_saturate(-1e9) == 0xFBFF
    assert oracle.f16_saturate(65519.0) == 0x7BFF
    assert oracle.f16_saturate(1.5) == 0x3E00


# --------------------------------------------------------------------------
# RHT: Sylvester closed form, orthogonality, exact inversion

@pytest.mark.parametrize("D", [2, 8, 64, 128])
def test_rht_equals_sylvester_closed_form(D):
    rng = np.random.default_rng(D)
    x = rng.integers(-50, 51, size=D).astype(np.float32)
    signs = np.where(rng.integers(0, 2, size=D) == 1, 1, -1).astype(np.int8)
    H = sylvester(D)
    want = H @ (signs.astype(np.int64) * x.astype(np.int64))  # exact integers
    got = oracle.rht_forward(x, signs)
    assert np.array_equal(got.astype(np.int64), want)
    assert np.array_equal(oracle.rht_forward(x, None).astype(np.int64), H @ x.astype(np.int64))


@pytest.mark.parametrize("D", [64, 128])
def test_rht_orthogonality_and_exact_inverse(D):
    H = sylvester(D)
    assert np.array_equal(H @ H.T, D * np.eye(D, dtype=np.int64))
    rng = np.random.default_rng(7)
    x = rng.integers(-100, 101, size=D).astype(np.float32)
    twice = oracle.rht_forward(oracle.rht_forward(x, None), None)
    assert np.array_equal(twice, D * x)


# --------------------------------------------------------------------------
# packing

def test_pack_round_trip_all_bytes():
    for mode, D in ((INT4, 64), (INT2, 128)):
        n = D // 2 if mode == INT4 else D // 4
        for b in range(256):
            data = np.full(n, b, dtype=np.uint8)
            codes = oracle.unpack_codes(mode, data, D)
            assert np.array_equal(oracle.pack_codes(mode, codes), data)


def test_pack_nibble_and_crumb_order():
    c4 = np.zeros(64, np.uint8)
    c4[0], c4[1] = 1, 2           # element 0 -> low nibble, element 1 -> high nibble
    assert oracle.pack_codes(INT4, c4)[0] == 0x21
    c2 = np.zeros(128, np.uint8)
    c2[:4] = [1, 2, 3, 0]         # element 4i+j -> bits 2j
    assert oracle.pack_codes(INT2, c2)[0] == 0b00111001


# --------------------------------------------------------------------------
# quantisation: worked grid rows, error bound, special cases

@pytest.mark.parametrize("mode,D", [(INT4, 64), (INT4, 128), (INT2, 64), (INT2, 128)])
def test_worked_grid_row_is_exact(mode, D):
    levels = 15 if mode == INT4 else 3
    s, m = 0.25, -1.5                       # powers of two / exact binary16 values
    k = np.arange(D) % (levels + 1)
    x = (m + s * k).astype(np.float32)
    row = oracle.quant_row(mode, x, None)
    data = D // 2 if mode == INT4 else D // 4
    if mode == INT4:
        want = (k[0::2] | (k[1::2] << 4)).astype(np.uint8)
        assert want[0] == 0x10 and want[1] == 0x32 and want[7] == 0xFE
    else:
        want = (k[0::4] | (k[1::4] << 2) | (k[2::4] << 4) | (k[3::4] << 6)).astype(np.uint8)
        assert want[0] == 0xE4
    assert np.array_equal(row[:data], want)
    S, M = f16_of_pad(row, data)
    assert (S, M) == (s, m)
    assert np.array_equal(oracle.dequant_row(mode, row, D), x.astype(np.float64))


@pytest.mark.parametrize("mode,D", [(INT4, 64), (INT4, 128), (INT2, 64), (INT2, 128)])
@pytest.mark.parametrize("rht", [False, True])
def test_ties_round_half_to_even_asymmetric(mode, D, rht):
    """Elements at M + (k + 1/2) S take the even code (tests/tie_rows.py);
    with the RHT on, the input is the exact pre-image of the same row."""
    y, codes = tie_rows.asym_row(4 if mode == INT4 else 2, D)
    signs = None
    x = y
    if rht:
        rng = np.random.default_rng(61 + D)
        signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8)
        x = tie_rows.pre_rotate(y, signs)
        assert np.array_equal(oracle.rht_forward(x, signs), y)
    row = oracle.quant_row(mode, x, signs)
    data = D // 2 if mode == INT4 else D // 4
    assert f16_of_pad(row, data) == (tie_rows.S_ASYM, tie_rows.M_ASYM)
    assert np.array_equal(oracle.unpack_codes(mode, row[:data], D), codes)
    if mode == INT4:
        assert row[:4].tolist() == [0xF0, 0x20, 0x42, 0x64]


@pytest.mark.parametrize("D", [64, 128])
def test_ties_round_half_to_even_stego(D):
    """Codes at t = k + 1/2 and a zero point at -lo / s = 2.5 both go to the
    even neighbour: zp = 2, pad 0x3E000002."""
    x, codes = tie_rows.stego_row(D)
    row = oracle.quant_row(STEGO, x, None)
    assert row[D // 2:D // 2 + 4].tolist() == tie_rows.STEGO_PAD
    assert stego_pad(row, D) == (tie_rows.S_STEGO, tie_rows.STEGO_ZP)
    assert np.array_equal(oracle.unpack_codes(STEGO, row[:D // 2], D), codes)
    assert row[:3].tolist() == [0xE0, 0x20, 0x42]


def test_ties_round_half_to_even_int8_channel():
    """Channel scales 2^(c % 7 - 3) fixed by an exact amax token; every later
    token sits at (j + 1/2) s_c and takes the even neighbour."""
    D = 64
    x, codes = tie_rows.int8_channel_tokens(D)
    T = x.shape[0]
    assert codes[:6, 0].tolist() == tie_rows.INT8_FIRST_CODES
    assert codes[-4:, 0].tolist() == tie_rows.INT8_LAST_CODES
    c, pg = _single_seq_paging(16, 16, T, INT8, D)
    assert oracle.write(c, pg, x[:, None, :], -x[:, None, :], np.array([0, T], np.int32)) == 0
    s = tie_rows.int8_channel_scales(D)
    assert np.array_equal(c.amax[0, 0], (127 * s).astype(np.float32))
    got_k = np.concatenate([c.k[blk, 0] for blk in range(16)])[:T].view(np.int8).astype(np.int64)
    got_v = np.concatenate([c.v[blk, 0] for blk in range(16)])[:T].view(np.int8).astype(np.int64)
    assert np.array_equal(got_k, codes)
    assert np.array_equal(got_v, -codes)      # rne is odd-symmetric: -t takes -rne(t)


@pytest.mark.parametrize("mode", [INT4, INT2])
@pytest.mark.parametrize("rht", [False, True])
def test_half_step_error_bound(mode, rht):
    D = 128
    rng = np.random.default_rng(3 + mode + 2 * rht)
    signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8) if rht else None
    levels = 15 if mode == INT4 else 3
    data = D // 2 if mode == INT4 else D // 4
    H = sylvester(D).astype(np.float64)
    for _ in range(200):
        x = (rng.standard_normal(D) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        x[rng.integers(0, D)] *= 20.0
        row = oracle.quant_row(mode, x, signs)
        S, M = f16_of_pad(row, data)
        xd = x.astype(np.float64)
        y = H @ (signs * xd) if rht else xd          # rotated row, closed form
        mn, mx = y.min(), y.max()
        s = (mx - mn) / levels
        slack = abs(mn - M) + levels * abs(s - S) + 1e-6 * max(abs(mn), abs(mx))
        xh = oracle.dequant_row(mode, row, D, signs)
        yh = H @ (signs * xh) if rht else xh          # back in the rotated domain
        assert np.max(np.abs(y - yh)) <= S / 2 + slack + 1e-9
        # in the input domain the l2 error shrinks by the RHT's norm sqrt(D)
        if rht:
            assert np.linalg.norm(xd - xh) <= (S / 2 + slack) * 1.0000001 + 1e-9
        codes = oracle.unpack_codes(mode, row[:data], D)
        assert codes.max() <= levels
        if S > 0 and slack < S / 2:
            assert codes[np.argmin(y)] == 0 and codes[np.argmax(y)] == levels


@pytest.mark.parametrize("mode", [INT4, INT2])
def test_constant_row_has_zero_scale(mode):
    D = 64
    x = np.full(D, 3.25, np.float32)
    row = oracle.quant_row(mode, x, None)
    data = D // 2 if mode == INT4 else D // 4
    assert np.all(row[:data] == 0)
    S, M = f16_of_pad(row, data)
    assert S == 0.0 and M == 3.25
    assert np.all(oracle.dequant_row(mode, row, D) == 3.25)


# ---------------------------------------------------------------------------
# INT4 with the zero point in the low 4 bits of an fp32 scale (vLLM PR #40835
# review summary, 评论区精华: zero-point steganography)

def stego_pad(row, D):
    w = int.from_bytes(bytes(row[D // 2:D // 2 + 4].tolist()), "little")
    return float(np.array([w & ~15], dtype=np.uint32).view(np.float32)[0]), w & 15


@pytest.mark.parametrize("D", [64, 128])
def test_stego_worked_grid_row_is_exact(D):
    k = np.arange(D) % 16
    x = ((k - 5) * 0.125).astype(np.float32)     # scale 2^-3, zero point 5
    row = oracle.quant_row(STEGO, x, None)
    want = (k[0::2] | (k[1::2] << 4)).astype(np.uint8)
    assert np.array_equal(row[:D // 2], want)
    # 0.125 is 0x3E000000; the zero point sits in the low 4 bits
    assert row[D // 2:D // 2 + 4].tolist() == [0x05, 0x00, 0x00, 0x3E]
    assert np.array_equal(oracle.dequant_row(STEGO, row, D), x.astype(np.float64))


@pytest.mark.parametrize("rht", [False, True])
def test_stego_error_bound(rht):
    """The grid (u - zp) s_t holds 0 and spans lo = min(min, 0) .. hi =
    max(max, 0): zp = rne(-lo / s_t) puts lo within half a step of the grid's
    bottom and hi within half a step plus the truncated scale bits of its top,
    so every value is within s_t / 2 + 15 (s - s_t) of its reconstruction
    (s = (hi - lo) / 15, s_t the stored scale)."""
    D = 128
    rng = np.random.default_rng(29 + rht)
    signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8) if rht else None
    H = sylvester(D).astype(np.float64)
    for _ in range(200):
        x = (rng.standard_normal(D) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        x[rng.integers(0, D)] *= 20.0
        row = oracle.quant_row(STEGO, x, signs)
        st, zp = stego_pad(row, D)
        xd = x.astype(np.float64)
        y = H @ (signs * xd) if rht else xd
        mn, mx = y.min(), y.max()
        lo, hi = min(mn, 0.0), max(mx, 0.0)
        s = (hi - lo) / 15
        assert 0 <= zp <= 15
        assert s * (1 - 4e-6) <= st <= s * (1 + 1e-6)    # 4 mantissa bits cleared
        xh = oracle.dequant_row(STEGO, row, D, signs)
        yh = H @ (signs * xh) if rht else xh
        bound = st / 2 + 15 * abs(s - st) + 2e-6 * max(abs(mn), abs(mx))
        assert np.max(np.abs(y - yh)) <= bound
        assert abs(lo - (-zp * st)) <= st / 2 + 2e-6 * max(abs(mn), abs(mx))


def test_stego_zero_constant_and_one_signed_rows():
    D = 64
    row = oracle.quant_row(STEGO, np.zeros(D, np.float32), None)
    assert np.all(row == 0)
    for c in (3.25, -3.25):                      # 15 steps between 0 and the value
        row = oracle.quant_row(STEGO, np.full(D, c, np.float32), None)
        st, zp = stego_pad(row, D)
        assert zp == (0 if c > 0 else 15)
        assert abs(15 * st - abs(c)) <= abs(c) * 2e-6
        xh = oracle.dequant_row(STEGO, row, D)
        assert np.max(np.abs(xh - c)) <= abs(c) * 2e-6
    x = np.linspace(2.0, 23.0, D).astype(np.float32)   # all positive: the grid still reaches the top
    row = oracle.quant_row(STEGO, x, None)
    st, zp = stego_pad(row, D)
    assert zp == 0 and np.max(np.abs(oracle.dequant_row(STEGO, row, D) - x)) <= st / 2 * 1.0001


# ---------------------------------------------------------------------------
# INT8 / FP8 with one symmetric scale per (token, kv head) (vLLM PR #40835
# review summary, 功能与动机 and 关联脉络: the per-token-head base modes)

def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(want)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_e4m3_round_matches_torch_incl_ties_subnormals_and_saturation():
    """torch's float32 -> float8_e4m3fn conversion rounds to nearest even; it
    agrees with the oracle wherever the result is finite (magnitudes below
    464).  Beyond that the oracle saturates at 448 (pattern 0x7E)."""
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])      # 0 .. 448, ascending
    mids = (vals[:-1] + vals[1:]) / 2                                   # every tie
    rng = np.random.default_rng(41)
    x = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
                        rng.uniform(0, 463.9, 4000), 2.0 ** rng.uniform(-14, 8.8, 4000)]).astype(np.float32)
    x = np.concatenate([x, -x])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, want)
    for v, c in ((448.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (470.0, 0x7E), (479.0, 0x7E), (1e6, 0x7E), (-500.0, 0xFE), (-0.0, 0x80)):
        assert oracle.e4m3_round(v) == c


def byte_pad(row, D):
    return float(np.frombuffer(bytes(row[D:D + 4].tolist()), dtype="<f4")[0])


def test_byte_token_head_worked_rows():
    """Hand-worked rows (RHT off) whose amax makes the scale exactly 1."""
    D = 64
    x = np.zeros(D, np.float32)
    x[:8] = [127, -63.5, 0.5, 1.5, 2.5, -2.5, -127, 3.0]
    row = oracle.quant_row(I8T, x, None)
    assert row[:8].view(np.int8).tolist() == [127, -64, 0, 2, 2, -2, -127, 3]   # ties to even
    assert np.all(row[8:D] == 0)
    assert row[D:].tolist() == [0x00, 0x00, 0x80, 0x3F]                          # fp32 1.0, little endian
    x = np.zeros(D, np.float32)
    x[:10] = [448, 1.0, 0.5, -2.0, 17.0, 19.0, 2.0 ** -9, 3 * 2.0 ** -10, -0.0, -448]
    row = oracle.quant_row(F8T, x, None)
    # 17 and 19 are ties (spacing 2 in [16, 32)): to 16 (fraction 000) and 20 (010)
    assert row[:10].tolist() == [0x7E, 0x38, 0x30, 0xC0, 0x58, 0x5A, 0x01, 0x02, 0x80, 0xFE]
    assert row[D:].tolist() == [0x00, 0x00, 0x80, 0x3F]
    assert oracle.dequant_row(F8T, row, D)[:10].tolist() == [448, 1, 0.5, -2, 16, 20, 2.0 ** -9, 2.0 ** -8, 0, -448]


@pytest.mark.parametrize("mode", [I8T, F8T])
@pytest.mark.parametrize("rht", [False, True])
def test_byte_token_head_error_bound(mode, rht):
    """In the rotated domain every element is within half a code step of its
    reconstruction: s / 2 for INT8; for FP8 half an E4M3 spacing of x / s,
    i.e. |y| 2^-4 above 2^-6 s and s 2^-10 below."""
    D = 128
    rng = np.random.default_rng(51 + mode + 2 * rht)
    signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8) if rht else None
    H = sylvester(D).astype(np.float64)
    for _ in range(200):
        x = (rng.standard_normal(D) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        x[rng.integers(0, D)] *= 20.0
        row = oracle.quant_row(mode, x, signs)
        xd = x.astype(np.float64)
        y = H @ (signs * xd) if rht else xd
        amax = np.abs(y).max()
        s = byte_pad(row, D)
        assert abs(s - amax / (127 if mode == I8T else 448)) <= 1e-6 * s
        xh = oracle.dequant_row(mode, row, D, signs)
        yh = H @ (signs * xh) if rht else xh
        err = np.abs(y - yh)
        slack = 2e-6 * amax
        if mode == I8T:
            assert err.max() <= s / 2 + slack
            codes = row[:D].view(np.int8).astype(int)
            assert np.abs(codes).max() == 127 and codes[np.argmax(np.abs(y))] == 127 * np.sign(y[np.argmax(np.abs(y))])
        else:
            assert np.all(err <= np.maximum(np.abs(y) * 2.0 ** -4, s * 2.0 ** -10) + slack)
            assert np.abs(oracle.dequant_row(mode, row, D)[:D]).max() <= 448 * s


@pytest.mark.parametrize("mode", [I8T, F8T])
def test_byte_token_head_zero_and_constant_rows(mode):
    D = 64
    row = oracle.quant_row(mode, np.zeros(D, np.float32), None)
    assert np.all(row == 0)
    for c in (3.25, -3.25):
        row = oracle.quant_row(mode, np.full(D, c, np.float32), None)
        want = {(I8T, True): 0x7F, (I8T, False): 0x81, (F8T, True): 0x7E, (F8T, False): 0xFE}[(mode, c > 0)]
        assert np.all(row[:D] == want)
        xh = oracle.dequant_row(mode, row, D)
        assert np.max(np.abs(xh - c)) <= abs(c) * 1e-6


def test_signed_zero_is_canonical():
    D = 64
    x = np.zeros(D, np.float32)
    x[::2] = -0.0
    row = oracle.quant_row(INT4, x, None)
    assert row[32:36].tolist() == [0, 0, 0, 0]


def _single_seq_paging(num_blocks, bs, T, mode, D, Hkv=1, signs=None):
    c = oracle.Cache(mode, num_blocks, Hkv, bs, D, signs)
    nb = (T + bs - 1) // bs
    table = np.arange(nb, dtype=np.int32)[None, :]
    pg = oracle.Paging(table, False, np.array([T], np.int32))
    return c, pg


def test_int8_per_channel_amax_symmetry_saturation():
    D, T = 64, 6
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, 1, D)).astype(np.float32)
    x[3] = -x[2]                                  # symmetric pair of tokens
    c, pg = _single_seq_paging(2, 16, T, INT8, D)
    assert oracle.write(c, pg, x, x * 0.5, np.array([0, T], np.int32)) == 0
    assert c.ready[0] == 1
    amax = np.abs(x[:, 0, :]).max(axis=0)
    assert np.array_equal(c.amax[0, 0], amax) and np.array_equal(c.amax[1, 0], amax * 0.5)
    q = c.k[0, 0, :T].view(np.int8).astype(np.int32)
    arg = np.abs(x[:, 0, :]).argmax(axis=0)
    assert np.all(np.abs(q[arg, np.arange(D)]) == 127)
    assert np.array_equal(q[3], -q[2])
    assert np.abs(q).max() <= 127
    # a later write reuses the frozen scales and saturates beyond them
    pg2 = oracle.Paging(pg.table, False, np.array([T + 1], np.int32))
    big = (x[:1] * 5.0).astype(np.float32)
    oracle.write(c, pg2, big, big, np.array([0, 1], np.int32))
    qb = c.k[0, 0, T].view(np.int8).astype(np.int32)
    assert np.array_equal(c.amax[0, 0], amax)
    assert np.all(qb[np.abs(big[0, 0]) >= amax * 1.01] ** 2 == 127 ** 2)


def test_int8_worked_grid_codes_and_dequant():
    """Channel c holds x = j * s_c for j in [-127, 127] with s_c a power of
    two: the amax is 127 s_c, the scale amax / 127 = s_c exactly, every code
    equals j and dequantisation returns x exactly."""
    D, T = 64, 255
    s = 2.0 ** (np.arange(D) % 7 - 3)
    j = np.arange(-127, 128)
    x = (j[:, None] * s[None, :]).astype(np.float32)[:, None, :]
    c, pg = _single_seq_paging(16, 16, T, INT8, D)
    assert oracle.write(c, pg, x, x, np.array([0, T], np.int32)) == 0
    assert np.array_equal(c.amax[0, 0], (127 * s).astype(np.float32))
    codes = np.concatenate([c.k[blk, 0] for blk in range(16)])[:T].view(np.int8).astype(np.int64)
    assert np.array_equal(codes, np.repeat(j[:, None], D, axis=1))
    row = c.k[0, 0, 5]
    assert np.array_equal(oracle.dequant_row(INT8, row, D, None, c.amax[0, 0]), x[5, 0].astype(np.float64))


# --------------------------------------------------------------------------
# attention: brute force on exact (grid) data, special cases, paging

def _grid_values(rng, n, D, mode):
    """Rows that INT4/INT2 (RHT off) or INT8 represent exactly."""
    if mode == INT8:
        return None
    if mode == I8T:  # j * s with s a power of two and |j| = 127 present
        j = rng.integers(-127, 128, size=(n, D))
        j[:, 0] = 127 * rng.choice([-1, 1], size=n)
        return (j * 2.0 ** rng.integers(-3, 2, size=(n, 1))).astype(np.float32)
    if mode == F8T:  # E4M3 values times a power of two, with 448 present
        c = rng.integers(0, 256, size=(n, D))
        c = np.where((c & 0x7F) == 0x7F, c - 1, c)                 # no NaN patterns
        e = np.array([oracle.e4m3_decode(i) for i in range(256)])
        v = e[c]
        v[:, 0] = 448 * rng.choice([-1, 1], size=n)
        return (v * 2.0 ** rng.integers(-3, 2, size=(n, 1))).astype(np.float32)
    if mode == STEGO:  # (k - zp) * s with s a power of two, min and max pinned
        k = rng.integers(0, 16, size=(n, D))
        k[:, 0], k[:, 1] = 0, 15
        s = 2.0 ** rng.integers(-3, 2, size=(n, 1))
        zp = rng.integers(0, 16, size=(n, 1))
        return ((k - zp) * s).astype(np.float32)
    levels = 15 if mode == INT4 else 3
    k = rng.integers(0, levels + 1, size=(n, D))
    k[:, 0], k[:, 1] = 0, levels                       # pin min and max of each row
    s = 2.0 ** rng.integers(-3, 2, size=(n, 1))
    m = -(2.0 ** rng.integers(-2, 3, size=(n, 1)))
    return (m + s * k).astype(np.float32)


def _softmax_ref(q, K, V, scale, mask):
    z = scale * (K @ q)
    z = np.where(mask, z, -np.inf)
    if not mask.any():
        return np.zeros(V.shape[1])
    p = np.exp(z - z.max())
    p /= p.sum()
    return p @ V


@pytest.mark.parametrize("mode", [INT4, INT2, STEGO, I8T, F8T])
def test_attention_brute_force_on_exact_rows(mode):
    rng = np.random.default_rng(11 + mode)
    D, bs, Hkv, Hq = 64, 16, 2, 4
    L = [23, 40]
    c = oracle.Cache(mode, 8, Hkv, bs, D)
    table = np.array([[5, 2, -1], [0, 7, 3]], np.int32)
    pg = oracle.Paging(table, False, np.array(L, np.int32))
    K = [_grid_values(rng, L[b] * Hkv, D, mode).reshape(L[b], Hkv, D) for b in range(2)]
    V = [_grid_values(rng, L[b] * Hkv, D, mode).reshape(L[b], Hkv, D) for b in range(2)]
    kk = np.concatenate(K)
    vv = np.concatenate(V)
    assert oracle.write(c, pg, kk, vv, np.array([0, L[0], L[0] + L[1]], np.int32)) == 0
    q = rng.standard_normal((2, Hq, D)).astype(np.float32)
    scale = 1.0 / math.sqrt(D)
    out, err = oracle.attention(c, pg, q, scale, threads=2)
    assert err == 0
    for b in range(2):
        for hq in range(Hq):
            h = hq // (Hq // Hkv)
            want = _softmax_ref(q[b, hq].astype(np.float64), K[b][:, h].astype(np.float64),
                                V[b][:, h].astype(np.float64), scale, np.ones(L[b], bool))
            np.testing.assert_allclose(out[b, hq], want, rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(2)
    D, bs = 64, 16
    c = oracle.Cache(INT4, 4, 1, bs, D)
    # single visible key -> its value row; equal keys -> mean of values
    kk = _grid_values(rng, 3, D, INT4)
    kk[1] = kk[0]
    kk[2] = kk[0]
    vv = _grid_values(rng, 3, D, INT4)
    pg = oracle.Paging(np.array([[1, -1]], np.int32), False, np.array([3], np.int32))
    oracle.write(c, pg, kk[:, None], vv[:, None], np.array([0, 3], np.int32))
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    out, _ = oracle.attention(c, pg, q, 0.125)
    np.testing.assert_allclose(out[0, 0], vv.astype(np.float64).mean(axis=0), rtol=0, atol=1e-12)
    pg1 = oracle.Paging(np.array([[1, -1]], np.int32), False, np.array([1], np.int32))
    out1, _ = oracle.attention(c, pg1, q, 0.125)
    assert np.array_equal(out1[0, 0], vv[0].astype(np.float64))
    # all keys evicted -> zero output
    pge = oracle.Paging(np.array([[-1, -1]], np.int32), False, np.array([3], np.int32))
    oute, _ = oracle.attention(c, pge, q, 0.125)
    assert np.all(oute == 0.0)


def test_write_skips_sentinel_and_flags_bad_ids():
    D, bs = 64, 16
    c = oracle.Cache(INT4, 4, 1, bs, D, fill=0xA5)
    x = np.ones((20, 1, D), np.float32)
    pg = oracle.Paging(np.array([[-1, 2]], np.int32), False, np.array([20], np.int32))
    assert oracle.write(c, pg, x, x, np.array([0, 20], np.int32)) == 0
    assert np.all(c.k[[0, 1, 3]] == 0xA5)              # block of the -1 entry untouched
    assert not np.all(c.k[2, 0, :4] == 0xA5)
    pgb = oracle.Paging(np.array([[9, 2]], np.int32), False, np.array([20], np.int32))
    assert oracle.write(c, pgb, x, x, np.array([0, 20], np.int32)) & 1
    pgt = oracle.Paging(np.array([[0]], np.int32), False, np.array([20], np.int32))
    assert oracle.write(c, pgt, x, x, np.array([0, 20], np.int32)) & 2
    assert oracle.write(c, pg, x, x, np.array([0, 20], np.int32)) == 0
    pgs = oracle.Paging(np.array([[0, 1]], np.int32), False, np.array([10], np.int32))
    assert oracle.write(c, pgs, x, x, np.array([0, 20], np.int32)) & 4


def test_evicted_blocks_do_not_contribute():
    rng = np.random.default_rng(4)
    D, bs, T = 64, 16, 64
    c = oracle.Cache(INT4, 8, 1, bs, D)
    kk = _grid_values(rng, T, D, INT4)[:, None]
    vv = _grid_values(rng, T, D, INT4)[:, None]
    full = oracle.Paging(np.array([[4, 5, 6, 7]], np.int32), False, np.array([T], np.int32))
    oracle.write(c, full, kk, vv, np.array([0, T], np.int32))
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    evict = oracle.Paging(np.array([[4, -1, -1, 7]], np.int32), False, np.array([T], np.int32))
    a, _ = oracle.attention(c, evict, q, 0.125)
    c.k[5:7] = rng.integers(0, 256, size=c.k[5:7].shape, dtype=np.uint8)   # garbage in evicted pages
    c.v[5:7] = rng.integers(0, 256, size=c.v[5:7].shape, dtype=np.uint8)
    b_, _ = oracle.attention(c, evict, q, 0.125)
    assert np.array_equal(a, b_)
    mask = np.zeros(T, bool)
    mask[:16] = True
    mask[48:] = True
    want = _softmax_ref(q[0, 0].astype(np.float64), kk[:, 0].astype(np.float64),
                        vv[:, 0].astype(np.float64), 0.125, mask)
    np.testing.assert_allclose(a[0, 0], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("W,sink", [(5, 0), (5, 3), (17, 2), (1, 0)])
def test_sliding_window_and_sink_visibility(W, sink):
    rng = np.random.default_rng(W * 10 + sink)
    D, bs, T, Hkv = 64, 16, 40, 2
    c = oracle.Cache(INT4, 4, Hkv, bs, D)
    kk = _grid_values(rng, T * Hkv, D, INT4).reshape(T, Hkv, D)
    vv = _grid_values(rng, T * Hkv, D, INT4).reshape(T, Hkv, D)
    pg = oracle.Paging(np.array([[0, 1, 2]], np.int32), False, np.array([T], np.int32),
                       window=np.array([0, W], np.int32), sink=sink)
    oracle.write(c, pg, kk, vv, np.array([0, T], np.int32))
    # prefill of the last 6 positions: each query has its own window
    n = 6
    q = rng.standard_normal((n, 2, D)).astype(np.float32)
    scale = float(np.float32(0.2))   # the oracle takes the scale as fp32
    out, _ = oracle.attention(c, pg, q, scale, cu_q=np.array([0, n], np.int32))
    for i in range(n):
        p = T - n + i
        j = np.arange(T)
        for h in range(Hkv):
            mask = j <= p
            if h == 1:
                mask &= (j < sink) | (j > p - W)
            want = _softmax_ref(q[i, h].astype(np.float64), kk[:, h].astype(np.float64),
                                vv[:, h].astype(np.float64), scale, mask)
            np.testing.assert_allclose(out[i, h], want, rtol=1e-12, atol=1e-12)


def test_headwise_table_rows_select_per_head_pages():
    """Row b * Hkv + h of a head-wise table serves (sequence b, kv head h)."""
    rng = np.random.default_rng(9)
    D, bs, T, Hkv, B = 64, 16, 20, 2, 2
    c = oracle.Cache(INT4, 10, Hkv, bs, D)
    kk = _grid_values(rng, B * T * Hkv, D, INT4).reshape(B * T, Hkv, D)
    vv = _grid_values(rng, B * T * Hkv, D, INT4).reshape(B * T, Hkv, D)
    rows = np.array([[0, 1], [2, 3], [4, 5], [6, 7]], np.int32)   # (b0,h0) (b0,h1) (b1,h0) (b1,h1)
    hw = oracle.Paging(rows, True, np.array([T, T], np.int32))
    oracle.write(c, hw, kk, vv, np.array([0, T, 2 * T], np.int32))
    # head 0 pages only in blocks 0,1,4,5; head 1 pages only in blocks 2,3,6,7
    assert np.all(c.k[[2, 3, 6, 7], 0] == 0) and np.all(c.k[[0, 1, 4, 5], 1] == 0)
    assert not np.all(c.k[4, 0] == 0) and not np.all(c.k[2, 1] == 0)
    q = rng.standard_normal((B, 2, D)).astype(np.float32)
    out, _ = oracle.attention(c, hw, q, 0.125)
    for b in range(B):
        for h in range(2):
            sl = slice(b * T, (b + 1) * T)
            want = _softmax_ref(q[b, h].astype(np.float64), kk[sl, h].astype(np.float64),
                                vv[sl, h].astype(np.float64), 0.125, np.ones(T, bool))
            np.testing.assert_allclose(out[b, h], want, rtol=1e-12, atol=1e-12)


def test_rht_attention_matches_brute_force_dequant():
    """With the RHT on, dequantised keys are d * (H y_hat) / D; check the
    oracle's attention against numpy with Sylvester's matrix and numpy's
    binary16 decoding of the stored scale and zero point."""
    wl = gen.tiny_int4(0)
    c = oracle.Cache(wl.mode, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.signs)
    pg = oracle.Paging(wl.table, False, wl.seq_lens)
    B, Hkv, D = wl.batch, wl.num_kv_heads, wl.head_dim
    kk = np.concatenate([gen.kv_values_host(wl, "k", b, 0, int(wl.seq_lens[b])) for b in range(B)])
    vv = np.concatenate([gen.kv_values_host(wl, "v", b, 0, int(wl.seq_lens[b])) for b in range(B)])
    assert oracle.write(c, pg, kk, vv, wl.cu(wl.seq_lens)) == 0
    q = gen.q_values_host(wl)
    out, err = oracle.attention(c, pg, q, 1.0 / math.sqrt(D))
    assert err == 0
    H = sylvester(D).astype(np.float64)
    sg = wl.signs.astype(np.float64)
    for b in range(B):
        L = int(wl.seq_lens[b])
        for hq in range(wl.num_q_heads):
            h = hq // wl.group
            Kh, Vh = np.zeros((L, D)), np.zeros((L, D))
            for j in range(L):
                blk = wl.table[b, j // 16]
                for dst, pages in ((Kh, c.k), (Vh, c.v)):
                    row = pages[blk, h, j % 16]
                    S, M = f16_of_pad(row, D // 2)
                    u = np.empty(D)
                    u[0::2] = row[:D // 2] & 15
                    u[1::2] = row[:D // 2] >> 4
                    dst[j] = sg * (H @ (u * S + M)) / D
            want = _softmax_ref(q[b, hq].astype(np.float64), Kh, Vh, 1.0 / math.sqrt(D), np.ones(L, bool))
            np.testing.assert_allclose(out[b, hq], want, rtol=1e-10, atol=1e-12)
    # and the quantisation error of the keys is within the half-step bound
    err_k = np.abs(Kh - kk[-L:, h].astype(np.float64)).max()
    assert err_k < 2.0


# ---------------------------------------------------------------------------
# gather and dequantise (FastDeploy PR #5173, the dynamic_quant_get_kv_from_cache
# op; Ascend INT8 plugin, 运行机制: prefill gathers and dequantises the pages)

def _rotated_grid_rows(rng, n, D, mode, signs):
    """Rows x whose RHT y = H (d * x) is a grid row of `mode`, built as x =
    d * (H y) / D with every partial sum exact in fp32, so that the write's
    fp32 butterfly recovers y exactly and the codes reproduce it."""
    if mode == F8T:   # E4M3 values that are multiples of 2^-3, 448 present
        e = np.array([oracle.e4m3_decode(i) for i in range(256)])
        ok = np.flatnonzero((np.abs(e) >= 1.0) & np.isfinite(e))
        y = e[rng.choice(ok, size=(n, D))]
        y[:, 0] = 448.0
    else:
        y = _grid_values(rng, n, D, mode).astype(np.float64)
    if signs is None:
        return y.astype(np.float32)
    H = sylvester(D).astype(np.float64)
    return ((y @ H) * signs[None, :] / D).astype(np.float32)


@pytest.mark.parametrize("mode", [INT4, INT2, STEGO, I8T, F8T])
@pytest.mark.parametrize("rht", [False, True])
def test_gather_round_trips_representable_rows_exactly(mode, rht):
    """Written then gathered, rows the mode represents exactly come back
    exactly, through scattered pages, a -1 entry (zero rows) and the write's
    position map (the last n_b positions of each sequence)."""
    rng = np.random.default_rng(61 + mode + 7 * rht)
    D, bs, Hkv = 64, 16, 2
    signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8) if rht else None
    L = [40, 23]
    c = oracle.Cache(mode, 9, Hkv, bs, D, signs, fill=0x5A)
    table = np.array([[6, -1, 3], [0, 8, -1]], np.int32)   # sequence 0's block 1 evicted
    pg = oracle.Paging(table, False, np.array(L, np.int32))
    x = [_rotated_grid_rows(rng, L[b] * Hkv, D, mode, signs).reshape(L[b], Hkv, D) for b in range(2)]
    w = [_rotated_grid_rows(rng, L[b] * Hkv, D, mode, signs).reshape(L[b], Hkv, D) for b in range(2)]
    assert oracle.write(c, pg, np.concatenate(x), np.concatenate(w), np.array([0, 40, 63], np.int32)) == 0
    # the last 30 positions of sequence 0 and all 23 of sequence 1
    k, v, err = oracle.gather(c, pg, np.array([0, 30, 53], np.int32))
    assert err == 0
    for b, (lo, t0) in enumerate(((10, 0), (0, 30))):
        n = L[b] - lo
        for i in range(n):
            p = lo + i
            want_k = np.zeros((Hkv, D)) if (b == 0 and 16 <= p < 32) else x[b][p].astype(np.float64)
            want_v = np.zeros((Hkv, D)) if (b == 0 and 16 <= p < 32) else w[b][p].astype(np.float64)
            assert np.array_equal(k[t0 + i], want_k), (b, p)
            assert np.array_equal(v[t0 + i], want_v), (b, p)


def test_gather_int8_channel_rows_and_errors():
    D, T = 64, 255
    s = 2.0 ** (np.arange(D) % 7 - 3)
    j = np.arange(-127, 128)
    x = (j[:, None] * s[None, :]).astype(np.float32)[:, None, :]
    c, pg = _single_seq_paging(16, 16, T, INT8, D)
    assert oracle.write(c, pg, x, -x, np.array([0, T], np.int32)) == 0
    k, v, err = oracle.gather(c, pg, np.array([0, T], np.int32))
    assert err == 0 and np.array_equal(k, x.astype(np.float64)) and np.array_equal(v, -x.astype(np.float64))
    # more tokens than the sequence holds, and a position past the table row
    _, _, err = oracle.gather(c, oracle.Paging(pg.table, False, np.array([3], np.int32)), np.array([0, 4], np.int32))
    assert err == 4
    k, _, err = oracle.gather(c, oracle.Paging(pg.table, False, np.array([T + 16], np.int32)),
                              np.array([0, T + 16], np.int32))
    assert err == 2 and np.all(k[T:] == 0)


# ---------------------------------------------------------------------------
# dense attention after a gather (the gather-then-dense-prefill strategy)

def _dense_paging(seq_lens, window=None, sink=0):
    B = len(seq_lens)
    return oracle.Paging(np.zeros((B, 1), np.int32), False, np.asarray(seq_lens, np.int32), window, sink)


@pytest.mark.parametrize("W,sink", [(0, 0), (9, 2)])
def test_dense_attention_brute_force(W, sink):
    """Causal prefill rows over dense K / V against a numpy brute force."""
    rng = np.random.default_rng(81 + W)
    D, Hkv, Hq = 64, 2, 4
    L, n = np.array([30, 12], np.int32), np.array([7, 12], np.int32)
    cu_kv = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    cu_q = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    k = rng.standard_normal((int(L.sum()), Hkv, D)).astype(np.float32)
    v = rng.standard_normal((int(L.sum()), Hkv, D)).astype(np.float32)
    q = rng.standard_normal((int(n.sum()), Hq, D)).astype(np.float32)
    win = np.array([0, W], np.int32) if W else None
    scale = 1.0 / math.sqrt(D)
    out, err = oracle.dense_attention(k, v, cu_kv, _dense_paging(L, win, sink), q, scale, cu_q, threads=2)
    assert err == 0
    for b in range(2):
        for i in range(n[b]):
            p = L[b] - n[b] + i
            for hq in range(Hq):
                h = hq // (Hq // Hkv)
                j = np.arange(L[b])
                mask = j <= p
                if win is not None and win[h] > 0:
                    mask &= (j < sink) | (j > p - win[h])
                want = _softmax_ref(q[cu_q[b] + i, hq].astype(np.float64), k[cu_kv[b]:cu_kv[b + 1], h].astype(np.float64),
                                    v[cu_kv[b]:cu_kv[b + 1], h].astype(np.float64), scale, mask)
                np.testing.assert_allclose(out[cu_q[b] + i, hq], want, rtol=1e-12, atol=1e-12)


def test_dense_attention_equals_paged_attention_on_exact_rows():
    """Rows INT8 token-head rows hold exactly (RHT off), given once as a paged
    cache and once as dense bf16 rows: both attentions agree."""
    rng = np.random.default_rng(83)
    D, bs, Hkv, Hq = 64, 16, 2, 4
    L = [40, 23]
    c = oracle.Cache(I8T, 9, Hkv, bs, D)
    table = np.array([[6, 2, 3], [0, 8, 5]], np.int32)
    pg = oracle.Paging(table, False, np.array(L, np.int32))
    x = [_grid_values(rng, L[b] * Hkv, D, I8T).reshape(L[b], Hkv, D) for b in range(2)]
    w = [_grid_values(rng, L[b] * Hkv, D, I8T).reshape(L[b], Hkv, D) for b in range(2)]
    kk, vv = np.concatenate(x), np.concatenate(w)
    assert oracle.write(c, pg, kk, vv, np.array([0, 40, 63], np.int32)) == 0
    q = rng.standard_normal((12, Hq, D)).astype(np.float32)
    cu_q = np.array([0, 5, 12], np.int32)
    scale = 0.125
    paged, err = oracle.attention(c, pg, q, scale, cu_q=cu_q, threads=2)
    assert err == 0
    kb, vb = gen.f32_to_bf16_bits(kk), gen.f32_to_bf16_bits(vv)   # exact: 8 significant bits suffice
    dense, err = oracle.dense_attention(kb, vb, np.array([0, 40, 63], np.int32), _dense_paging(L), q, scale, cu_q,
                                        threads=2)
    assert err == 0
    np.testing.assert_allclose(dense, paged, rtol=1e-12, atol=1e-12)
    # a cu_kv that disagrees with seq_lens is refused
    _, err = oracle.dense_attention(kb, vb, np.array([0, 39, 63], np.int32), _dense_paging(L), q, scale, cu_q)
    assert err == 4


def test_gather_with_full_precision_chunk():
    """The chunk positions come back exactly as given (fp32 and bf16 rows);
    the earlier positions as the plain gather gives them; a chunk longer than
    its sequence is flagged."""
    rng = np.random.default_rng(87)
    D, bs, Hkv = 64, 16, 2
    L, m = np.array([40, 23], np.int32), np.array([10, 23], np.int32)
    signs = np.where(rng.integers(0, 2, D) == 1, 1, -1).astype(np.int8)
    c = oracle.Cache(INT4, 9, Hkv, bs, D, signs)
    pg = oracle.Paging(np.array([[6, 2, 3], [0, 8, 5]], np.int32), False, L)
    x = rng.standard_normal((63, Hkv, D)).astype(np.float32)
    assert oracle.write(c, pg, x, -x, np.array([0, 40, 63], np.int32)) == 0
    chunk = rng.standard_normal((int(m.sum()), Hkv, D)).astype(np.float32)
    cu_chunk = np.array([0, 10, 33], np.int32)
    cu_all = np.array([0, 40, 63], np.int32)
    for ck in (chunk, gen.f32_to_bf16_bits(chunk)):
        k, v, err = oracle.gather_chunk(c, pg, cu_all, ck, ck, cu_chunk)
        assert err == 0
        want = chunk if ck.dtype == np.float32 else gen.bf16_bits_to_f32(ck)
        assert np.array_equal(k[30:40], want[0:10].astype(np.float64))
        assert np.array_equal(v[40:63], want[10:33].astype(np.float64))
        kp, vp, _ = oracle.gather(c, pg, cu_all)
        assert np.array_equal(k[:30], kp[:30]) and np.array_equal(v[:30], vp[:30])
    _, _, err = oracle.gather_chunk(c, pg, cu_all, chunk, chunk, np.array([0, 10, 40], np.int32))
    assert err == 4
