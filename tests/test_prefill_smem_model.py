"""A host-side model of the chunked-prefill kernel's shared-memory loads.

For one 64-key tile of the INT4, head_dim 128 prefill (prefill_tc_kernel),
each role's warp-level shared loads are replayed from the kernel's own index
arithmetic (lane -> byte address and width), and their wavefronts are counted
with the bank rule: 32 banks of 4 bytes; a 4-byte or narrower access is one
phase; an 8-byte access two phases of 16 lanes and a 16-byte access four
phases of 8 lanes; in a phase, the wavefronts are the largest number of
distinct 4-byte words any one bank is asked for (lanes reading the same word
share it).  A load's conflict wavefronts are those beyond its phases.

The model locates every excess wavefront per tile in one place, the
producers' key expansion: with 68-byte (17-word) rows, the last code word of
key k + 1 lands in the bank of the first code word of key k, so each of its
32 loads per tile is 2-way.  The value expansion, the scale / zero-point reads and the softmax's
scale reads (the same 16 bytes in every lane) are conflict-free under the
rule.  The measured counts, and how they compare, are in the prefill profile
summary.

For the dense bf16 rows of the same kernel the value expansion reads one
column of eight 256-byte rows at a time, all in one bank (8-way); the tensor
copies therefore land each 64-dim half with the 128-byte swizzle, which the
model shows conflict-free for both expansions.
"""
from collections import defaultdict

TP_KT = 64           # keys per tile
D = 128
R = D // 2 + 4       # INT4 row bytes
DATA = D // 2
TP_PRODUCERS = 128   # 4 producer warps
KSTEP = TP_PRODUCERS // (D // 8)


def wavefronts(addrs, width):
    """Wavefronts of one warp-level shared load: addrs[lane] (bytes), width in bytes."""
    phases = max(1, width // 4)
    lanes_per_phase = 32 // phases
    total = 0
    for ph in range(phases):
        words_by_bank = defaultdict(set)
        for lane in range(ph * lanes_per_phase, (ph + 1) * lanes_per_phase):
            a = addrs[lane]
            if a is None:
                continue
            for w in range(max(1, width // 4)):
                word = a // 4 + w
                words_by_bank[word % 32].add(word)
        total += max((len(s) for s in words_by_bank.values()), default=0)
    return total, phases


def key_expansion_loads():
    """Producer warp pw, item j: lds32(rk + (key_0 + KSTEP j) R + 4 c8),
    thread pt = 32 pw + lane: c8 = pt % (D/8), key_0 = pt / (D/8)."""
    out = []
    for pw in range(4):
        for j in range(TP_KT * (D // 8) // TP_PRODUCERS):
            addrs = []
            for lane in range(32):
                pt = 32 * pw + lane
                c8, key_0 = pt % (D // 8), pt // (D // 8)
                addrs.append((key_0 + KSTEP * j) * R + 4 * c8)
            out.append((addrs, 4))
    return out


def value_expansion_loads():
    """Producer warp pw, job pw + 4 jj: lane (g8, t4) reads byte
    rvp + (8 kb + g8) R + (32 db + 8 i + 2 t4) / 2 for i = 0..3."""
    out = []
    jobs = (TP_KT // 8) * (D // 32)
    for pw in range(4):
        for jj in range(jobs // 4):
            job = pw + 4 * jj
            kb, db = job % (TP_KT // 8), job // (TP_KT // 8)
            for i in range(4):
                addrs = []
                for lane in range(32):
                    g8, t4 = lane >> 2, lane & 3
                    addrs.append((8 * kb + g8) * R + (32 * db + 8 * i + 2 * t4) // 2)
                out.append((addrs, 1))
    return out


def scale_pad_loads():
    """Producer thread pt reads the pad of key pt & 63 (K rows for pt < 64, V rows after)."""
    out = []
    for pw in range(4):
        addrs = []
        for lane in range(32):
            idx = 32 * pw + lane
            key, isv = idx & (TP_KT - 1), idx >= TP_KT
            addrs.append((TP_KT * R if isv else 0) + key * R + DATA)
        out.append((addrs, 4))
    return out


def softmax_scale_loads():
    """Softmax warp (quad, half hf): for chunks c = 2 hf, 2 hf + 1 and j4 = 0..3,
    float4 reads of ks, kz (pass 1) and vs, vz (pass 2) at the same address in
    every lane: 32 per warp per tile, 8 warps."""
    out = []
    for w in range(8):
        hf = w >> 2
        for c in (2 * hf, 2 * hf + 1):
            for j4 in range(4):
                for arr in range(4):  # ks, kz, vs, vz: 16 float4 each
                    a = 16 * (16 * arr + 4 * c + j4)
                    out.append(([a] * 32, 16))
    return out


def dense_vt_loads(swizzled):
    """Dense rows (bf16, 2 D bytes), value expansion: producer job (kb, db),
    lane (g8, t4) reads the 4 bytes of dims 32 db + 8 i + 2 t4 and + 1 of key
    row 8 kb + g8, i = 0..3.  Unswizzled the rows are 256 bytes apart; the
    kernel's tensor copies instead land each 64-dim half as 64 lines of 128
    bytes with 16-byte piece c of line r at piece c ^ (r & 7)."""
    out = []
    for kb in range(TP_KT // 8):
        for db in range(D // 32):
            for i in range(4):
                addrs = []
                for lane in range(32):
                    g8, t4 = lane >> 2, lane & 3
                    addrs.append(dense_addr(8 * kb + g8, 32 * db + 8 * i + 2 * t4, swizzled))
                out.append((addrs, 4))
    return out


def dense_addr(row, d, swizzled):
    if not swizzled:
        return row * 2 * D + 2 * d
    c = (d % 64) // 8
    return (d // 64) * 64 * 128 + row * 128 + 16 * (c ^ (row & 7)) + 2 * (d % 8)


def role_totals(loads):
    waves = phases = instr = 0
    for addrs, width in loads:
        wv, ph = wavefronts(addrs, width)
        waves += wv
        phases += ph
        instr += 1
    return instr, waves, waves - phases


def test_key_expansion_is_two_way():
    instr, waves, excess = role_totals(key_expansion_loads())
    assert instr == 32 and waves == 64 and excess == 32
    # the colliding pair: lane 0 (first code word of key k) and lane 31 (last
    # code word of key k + 1), 17 + 15 = 32 words apart
    addrs, _ = key_expansion_loads()[0]
    banks = [(a // 4) % 32 for a in addrs]
    assert banks[0] == banks[31] and len(set(banks)) == 31


def test_value_expansion_and_pads_are_conflict_free():
    assert role_totals(value_expansion_loads()) == (128, 128, 0)
    assert role_totals(scale_pad_loads()) == (4, 4, 0)


def test_softmax_scale_reads_are_broadcasts():
    instr, waves, excess = role_totals(softmax_scale_loads())
    assert instr == 256 and excess == 0
    # under the rule each broadcast float4 still takes its four phases
    assert waves == 4 * 256


def test_wavefront_rule_on_textbook_patterns():
    assert wavefronts([4 * l for l in range(32)], 4) == (1, 1)            # consecutive words
    assert wavefronts([128 * l for l in range(32)], 4) == (32, 1)         # one bank, 32 words
    assert wavefronts([0] * 32, 4) == (1, 1)                              # broadcast
    assert wavefronts([16 * l for l in range(32)], 16) == (4, 4)          # 512 contiguous bytes
    assert wavefronts([8 * (l % 16) * 2 for l in range(32)], 8) == (4, 2)  # 2-way in each half


def test_dense_value_expansion_swizzle():
    # 256-byte rows put one column of eight rows in one bank: every load 8-way
    instr, waves, excess = role_totals(dense_vt_loads(False))
    assert instr == 128 and excess == 7 * instr
    # the 128-byte swizzle of the tensor copies spreads them over all banks
    assert role_totals(dense_vt_loads(True)) == (128, 128, 0)
    # and the swizzled layout is still one place per (row, dim pair): a
    # permutation of the tile's 4-byte words
    words = {dense_addr(r, d, True) // 4 for r in range(TP_KT) for d in range(0, D, 2)}
    assert words == set(range(TP_KT * D // 2))


def test_dense_key_expansion_swizzled_reads_conflict_free():
    # producer thread pt reads 16 bytes (dims 8 c8 .. 8 c8 + 7) of key row
    # pt / (D/8) + KSTEP j: whole pieces, so the piece index is swizzled
    loads = []
    for pw in range(4):
        for j in range(TP_KT * (D // 8) // TP_PRODUCERS):
            addrs = []
            for lane in range(32):
                pt = 32 * pw + lane
                c8, key = pt % (D // 8), pt // (D // 8) + KSTEP * j
                addrs.append(dense_addr(key, 8 * c8, True))
            loads.append((addrs, 16))
    instr, waves, excess = role_totals(loads)
    assert excess == 0
