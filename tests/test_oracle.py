"""Pins for the W12 oracle: checks against facts that do not come from the oracle.

- lossless / bit-exact ("StargazerX0/SpecPilot" §What it is; "SpecPilot"
  §Differentiation): every BF16 bit pattern survives encode -> decode;
- a hand-worked 2x2 blob fixes the byte layout;
- the exponent table is a top-15 set and the escapes are exactly the histogram
  mass outside it;
- Gaussian weights: bits/weight close to 12 ("SpecPilot: an agent doubled ..."
  §The mechanisms it found) and an escape rate matching the normal CDF;
- the fp64 GEMM against numpy's float64 matmul and exact special cases.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from lossless_bit_weight_encode_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def _hdr(blob, off, n):
    return int.from_bytes(bytes(blob[off:off + n]), "little")


def _seg_headers(blob):
    off, nbytes = _hdr(blob, 0x58, 8), _hdr(blob, 0x60, 8)
    return np.asarray(blob[off:off + nbytes]).reshape(-1, 32)


def _padded(w):
    n, k = w.shape
    npad, kpad = -(-n // 128) * 128, -(-k // 32) * 32
    out = np.zeros((npad, kpad), dtype=np.uint16)
    out[:n, :k] = w
    return out


@pytest.mark.parametrize("shuffle", [None, 1, 2, 3])
def test_exhaustive_bf16_round_trip(shuffle):
    w = wl.all_bf16_patterns(shuffle)
    assert np.array_equal(oracle.decode(oracle.encode(w)), w)


@pytest.mark.parametrize("shape", [(128, 512), (512, 128), (64, 1024), (1000, 70), (3, 21845)])
def test_exhaustive_patterns_other_shapes(shape):
    v = wl.all_bf16_patterns(5).reshape(-1)
    n, k = shape
    w = np.resize(v, n * k).reshape(n, k)
    assert np.array_equal(oracle.decode(oracle.encode(w)), w)


@pytest.mark.parametrize("shape", [(1, 1), (1, 33), (129, 31), (127, 257), (300, 1000)])
def test_ragged_round_trip(shape):
    w = wl.gaussian_weights(*shape, seed=11)
    assert np.array_equal(oracle.decode(oracle.encode(w)), w)


def test_special_groups_round_trip():
    rng = np.random.default_rng(3)
    # one exponent everywhere
    one = ((rng.integers(0, 2, (256, 512)) << 15) | (120 << 7) | rng.integers(0, 128, (256, 512))).astype(np.uint16)
    # exactly 16 distinct exponents -> exactly one exponent escapes per segment
    e16 = rng.integers(100, 116, (256, 512))
    sixteen = ((e16 << 7) | rng.integers(0, 128, (256, 512))).astype(np.uint16)
    # every weight escapes: 256 exponents in equal shares, most outside any table
    allesc = wl.forced_escape_weights(256, 512, 1.0, seed=4)
    for w in (one, sixteen, allesc):
        assert np.array_equal(oracle.decode(oracle.encode(w)), w)
    blob = oracle.encode(one)
    assert _hdr(blob, 0x80, 8) == 0
    blob16 = oracle.encode(sixteen)
    assert _hdr(blob16, 0x80, 8) > 0


def test_hand_worked_2x2_blob():
    # W = [[1.0, -2.0], [0.5, 3.0]] padded with +0.0 to 128 x 32.
    # exponents: 1.0 -> 127, -2.0 -> 128, 0.5 -> 126, 3.0 -> 128, pads -> 0.
    # counts: 0:4092, 128:2, 126:1, 127:1; ranked 0, 128, 126, 127.
    # L = [0, 126, 127] (odd), H = [128]: sequence 0, 126, 127, 128 into the
    # slots 7, 0, 8, 1; slot 9 copies its partner 1; the rest are 0.
    w = np.array([[0x3F80, 0xC000], [0x3F00, 0x4040]], dtype=np.uint16)
    blob = oracle.encode(w)
    assert bytes(blob[:4]) == b"W12B"
    assert _hdr(blob, 0x04, 4) == 1 and _hdr(blob, 0x10, 8) == 2 and _hdr(blob, 0x18, 8) == 2
    assert _hdr(blob, 0x20, 8) == 128 and _hdr(blob, 0x28, 8) == 32
    assert _hdr(blob, 0x40, 8) == 1 and _hdr(blob, 0x48, 8) == 1 and _hdr(blob, 0x50, 8) == 1
    assert _hdr(blob, 0x58, 8) == 256 and _hdr(blob, 0x60, 8) == 32
    assert _hdr(blob, 0x68, 8) == 512 and _hdr(blob, 0x70, 8) == 6144
    assert _hdr(blob, 0x78, 8) == 512 + 6144 and _hdr(blob, 0x80, 8) == 0
    assert _hdr(blob, 0x90, 8) == blob.size == 512 + 6144
    table = list(blob[256:272])
    assert table == [126, 128, 0, 0, 0, 0, 0, 0, 127, 128, 0, 0, 0, 0, 0, 0]
    assert list(blob[272:304]) == [0] * 32  # no escapes: base 0, counts 0, mask 0
    chunk = blob[512:512 + 6144]
    # S bytes: (mantissa << 1) | sign of the pair partner
    assert chunk[0] == 1 and chunk[1] == 0          # 1.0 takes -2.0's sign; -2.0 takes 1.0's
    assert chunk[16] == 0 and chunk[17] == 0x80     # 3.0 has mantissa 0x40
    assert np.count_nonzero(chunk[:4096]) == 2
    # codes: 127 -> 8, 128 -> 1, 126 -> 0; the pad exponent 0 first appears at slot 2
    assert chunk[4096] == 0x18 and chunk[4096 + 16] == 0x10
    codes = np.array(chunk[4096:]).reshape(128, 16)
    codes[0, 0] = codes[1, 0] = 0x22
    assert np.all(codes == 0x22)
    assert np.array_equal(oracle.decode(blob), w)


def _check_tables(w, blob):
    wp = _padded(w)
    expo = (wp >> 7) & 0xFF
    heads = _seg_headers(blob)
    tiles, segs = wp.shape[0] // 128, -(-wp.shape[1] // 256)
    n_esc = 0
    for t in range(tiles):
        for s in range(segs):
            hd = heads[t * segs + s]
            T = hd[:16]
            assert T[15] == 0
            for j in range(7):
                assert (T[j] >> 7) == (T[j + 8] >> 7), "pair slots must share the top bit"
            blk = expo[128 * t:128 * (t + 1), 256 * s:256 * (s + 1)]
            hist = np.bincount(blk.reshape(-1), minlength=256)
            present = [e for e in range(256) if hist[e] > 0]
            ranked = sorted(present, key=lambda e: (-hist[e], e))[:15]
            held = set(int(v) for v in T[:15])
            assert set(ranked) <= held
            assert held - set(ranked) <= {0}
            esc = int(sum(hist[e] for e in range(256) if e not in held))
            qcount = [int(hd[20 + 2 * q]) | (int(hd[21 + 2 * q]) << 8) for q in range(4)]
            assert sum(qcount) == esc
            for q in range(4):
                qb = blk[32 * q:32 * (q + 1)]
                assert qcount[q] == int(sum(np.count_nonzero(qb == e) for e in range(256) if e not in held))
            mask = int.from_bytes(bytes(hd[28:32]), "little")
            for q in range(4):
                for j in range(8):
                    cb = blk[32 * q:32 * (q + 1), 32 * j:32 * (j + 1)]
                    has = any(np.count_nonzero(cb == e) for e in range(256) if e not in held)
                    assert bool(mask >> (8 * q + j) & 1) == has
            base = int.from_bytes(bytes(hd[16:20]), "little")
            assert base == n_esc
            n_esc += esc
    assert n_esc == _hdr(blob, 0x80, 8)


@pytest.mark.parametrize("kind", ["gauss", "heavy", "forced2", "forced10", "allbits"])
def test_table_is_top15_and_escapes_are_outside_mass(kind):
    if kind == "gauss":
        w = wl.gaussian_weights(256, 700, seed=21)
    elif kind == "heavy":
        w = wl.heavy_tail_weights(256, 700, seed=22)
    elif kind == "forced2":
        w = wl.forced_escape_weights(200, 600, 0.02, seed=23)
    elif kind == "forced10":
        w = wl.forced_escape_weights(200, 600, 0.10, seed=24)
    else:
        w = wl.all_bf16_patterns(9)
    _check_tables(w, oracle.encode(w))


def _expected_size(n, k, n_esc):
    up = lambda v, a: -(-v // a) * a
    tiles, chunks = up(n, 128) // 128, up(k, 32) // 32
    segs = -(-chunks // 8)
    off_w = up(256 + 32 * tiles * segs, 256)
    off_e = up(off_w + 6144 * tiles * chunks, 256)
    return up(off_e + up(n_esc, 16), 256)


@pytest.mark.parametrize("shape", [(1, 1), (128, 32), (130, 300), (1024, 1024)])
def test_size_closed_form(shape):
    w = wl.forced_escape_weights(*shape, 0.01, seed=5)
    blob = oracle.encode(w)
    assert blob.size == oracle.encoded_size(w) == _expected_size(*shape, _hdr(blob, 0x80, 8))


def _gaussian_bin_mass(std):
    """P(BF16(N(0, std)) has biased exponent e), from the normal CDF; the lower
    edge of bin e is the midpoint between 2^(e-127) and its BF16 predecessor."""
    def cdf_abs(v):
        return math.erf(v / (std * math.sqrt(2.0)))
    edges = {}
    for e in range(1, 256):
        p2 = 2.0 ** (e - 127)
        edges[e] = p2 - 2.0 ** (e - 127 - 9)
    mass = {}
    for e in range(1, 255):
        mass[e] = cdf_abs(edges[e + 1]) - cdf_abs(edges[e])
    mass[0] = cdf_abs(edges[1])
    return mass


def test_gaussian_escape_rate_matches_normal_cdf():
    w = wl.gaussian_weights(2048, 4096, seed=31)
    blob = oracle.encode(w)
    n_esc = _hdr(blob, 0x80, 8)
    mass = _gaussian_bin_mass(wl.WEIGHT_STD)
    top = sorted(mass, key=lambda e: -mass[e])[:15]
    expect = (1.0 - sum(mass[e] for e in top)) * w.size
    assert abs(n_esc - expect) < 0.15 * expect + 5 * math.sqrt(expect)


def test_bits_per_weight_near_twelve():
    w, _ = wl.single_case()
    bpw = 8.0 * oracle.encoded_size(w) / w.size
    facts = FACTS["bits_per_weight_dense"]
    assert 12.0 < bpw <= facts["high"] + 0.005
    big = wl.gaussian_weights(2048, 4096, seed=32)
    bpw_big = 8.0 * oracle.encoded_size(big) / big.size
    assert 12.0 < bpw_big <= facts["high"]
    # "cuts weight traffic by a quarter": packed bytes / BF16 bytes
    ratio = oracle.encoded_size(big) / (2.0 * big.size)
    assert abs(ratio - (1.0 - FACTS["weight_traffic_cut"]["value"])) < 0.002


def test_gemm_f64_matches_numpy_float64():
    rng = np.random.default_rng(7)
    for m, n, k in [(1, 5, 7), (3, 33, 65), (32, 130, 257)]:
        x = wl.activations(m, k, seed=int(rng.integers(1 << 30)))
        w = wl.gaussian_weights(n, k, seed=int(rng.integers(1 << 30)))
        ref = wl.bf16_bits_to_f32(x).astype(np.float64) @ wl.bf16_bits_to_f32(w).astype(np.float64).T
        assert np.allclose(oracle.gemm_f64(x, w), ref, rtol=1e-12, atol=1e-12)


def test_gemm_f64_one_hot_and_small_integers():
    w = wl.gaussian_weights(64, 48, seed=8)
    for kk in (0, 17, 47):
        x = np.zeros((1, 48), dtype=np.uint16)
        x[0, kk] = 0x3F80  # 1.0
        y = oracle.gemm_f64(x, w)
        assert np.array_equal(y[0], wl.bf16_bits_to_f32(w[:, kk]).astype(np.float64))
    rng = np.random.default_rng(9)
    wi = rng.integers(-8, 9, (40, 100))
    xi = rng.integers(-8, 9, (4, 100))
    y = oracle.gemm_f64(wl.to_bf16_bits(xi.astype(np.float32)), wl.to_bf16_bits(wi.astype(np.float32)))
    assert np.array_equal(y, (xi @ wi.T).astype(np.float64))


def test_w12_gemm_equals_gemm_over_original():
    w = wl.heavy_tail_weights(300, 520, seed=10)
    x = wl.activations(5, 520, seed=11)
    blob = oracle.encode(w)
    assert np.array_equal(oracle.w12_gemm_f64(x, blob, threads=2), oracle.gemm_f64(x, w))


def test_malformed_blobs_are_rejected():
    w = wl.gaussian_weights(130, 70, seed=12)
    blob = oracle.encode(w)
    with pytest.raises(ValueError):
        oracle.decode(blob[:-256])
    bad = blob.copy()
    bad[0] = ord("X")
    with pytest.raises(ValueError):
        oracle.decode(bad)
    bad = blob.copy()
    bad[0x11] ^= 1  # N grows by 256: padded geometry no longer matches
    with pytest.raises(ValueError):
        oracle.decode(bad)


def test_argmax_f64_ties_nan_and_brute_force():
    """The LM-head argmax restated: lowest index among equal maxima, NaN
    logits never chosen, and agreement with an explicit scan on small cases."""
    one = np.uint16(0x3F80)  # 1.0
    w = np.zeros((6, 4), dtype=np.uint16)
    w[1, 0] = w[4, 0] = np.uint16(0x4000)  # 2.0 in rows 1 and 4: a tie
    w[2, 1] = np.uint16(0x7FC0)            # NaN
    w[3, 1] = np.uint16(0xBF80)            # -1.0
    x = np.zeros((2, 4), dtype=np.uint16)
    x[0, 0] = one
    x[1, 1] = one
    idx, y = oracle.argmax_f64(x, w)
    assert idx[0] == 1                      # tie between rows 1 and 4
    assert np.isnan(y[1, 2]) and idx[1] == 0  # NaN ranks below 0.0 and -1.0 is below 0.0
    rng = np.random.default_rng(13)
    for trial in range(5):
        w = wl.to_bf16_bits(rng.integers(-3, 4, (50, 30)).astype(np.float32))
        x = wl.to_bf16_bits(rng.integers(-3, 4, (3, 30)).astype(np.float32))
        idx, y = oracle.argmax_f64(x, w)
        for m in range(3):
            best, arg = -np.inf, -1
            for n in range(50):
                if y[m, n] > best:
                    best, arg = y[m, n], n
            assert idx[m] == arg


def test_q8_hand_worked_row():
    """Row maximum 127/64 makes the scale exactly 1/64, so q = rint(64 w) can
    be worked by hand: 32.5 -> 32 and 33.5 -> 34 (ties to even)."""
    vals = np.array([127 / 64, 32.5 / 64, 33.5 / 64, -32.5 / 64, 0.0, -127 / 64, 1 / 128, 3 / 128],
                    dtype=np.float32)
    w = wl.to_bf16_bits(vals[None, :])
    assert np.array_equal(wl.bf16_bits_to_f32(w)[0], vals)  # all exact in BF16
    s, q = oracle.q8_decode(oracle.q8_encode(w), 1, 8)
    assert s[0] == np.float32(1 / 64)
    assert q[0].tolist() == [127, 32, 34, -32, 0, -127, 0, 2]  # 0.5 -> 0 and 1.5 -> 2: ties to even


def test_q8_invariants_and_layout():
    rng = np.random.default_rng(14)
    w = wl.heavy_tail_weights(300, 333, seed=15)
    w[7] = 0  # a zero row
    s, q = oracle.q8_decode(oracle.q8_encode(w), 300, 333)
    wf = wl.bf16_bits_to_f32(w).astype(np.float64)
    nz = np.abs(wf).max(axis=1) > 0
    assert np.all(np.abs(q).max(axis=1)[nz] == 127) and s[7] == 0 and not q[7].any()
    # each entry within half a step of its weight (plus the fp32 rounding of s)
    err = np.abs(wf - s.astype(np.float64)[:, None] * q)
    assert np.all(err <= 0.5 * s.astype(np.float64)[:, None] * (1 + 1e-5) + 1e-30)
    # byte position of (n=129, k=40): tile 1, chunk 1, slab 0 (column 8), row 1
    w2 = np.zeros((130, 64), dtype=np.uint16)
    w2[129, 40] = np.uint16(0xBF80)  # -1.0
    b = oracle.q8_encode(w2)
    off_q = int(b[0x50:0x58].view(np.uint64)[0])
    chunks = 2
    assert b[off_q + 4096 * (1 * chunks + 1) + 16 * 1 + 8] == np.uint8(256 - 127)
    assert int(np.count_nonzero(b[off_q:])) == 1
    assert b[:4].tobytes() == b"Q8W1"
    bad = w.copy()
    bad[3, 3] = np.uint16(0x7F80)  # +Inf
    with pytest.raises(ValueError):
        oracle.q8_encode(bad)
    del rng


def test_q8_gemm_hand_worked_products():
    """oracle.q8_gemm_f64 against products worked by hand.  Row 0 has maximum
    127/64, so its scale is exactly 1/64 and q = [127, 32, 34, -32, 0, -127,
    0, 2] (as in the row above); row 1 has maximum 127/32 (scale 1/32) and
    values 1/32, 2.5/32 and 3.5/32, so q = [1, -127, 2, 4, 0, 0, 0, 0] (2.5
    ties to 2, 3.5 to 4).  A one-hot x picks s[n] q[n, k]; a small-integer x
    gives sums that are worked out below."""
    r0 = [127 / 64, 32.5 / 64, 33.5 / 64, -32.5 / 64, 0.0, -127 / 64, 1 / 128, 3 / 128]
    r1 = [1 / 32, -127 / 32, 2.5 / 32, 3.5 / 32, 0.0, 0.0, 0.0, 0.0]
    w = wl.to_bf16_bits(np.array([r0, r1], dtype=np.float32))
    # one-hot x: column k of s q, i.e. q[n, k] / 64 and q[n, k] / 32
    x = np.zeros((3, 8), dtype=np.uint16)
    x[0, 1] = x[1, 3] = x[2, 5] = np.uint16(0x3F80)  # 1.0
    y = oracle.q8_gemm_f64(x, w)
    assert y.tolist() == [[32 / 64, -127 / 32], [-32 / 64, 4 / 32], [-127 / 64, 0.0]]
    # x = [1, 2, 0, -1, 3, 1, 5, -2]:
    #   row 0: 127 + 64 + 0 + 32 + 0 - 127 + 0 - 4 = 92   -> 92 / 64
    #   row 1: 1 - 254 + 0 - 4 + 0 + 0 + 0 + 0 = -257     -> -257 / 32
    # x = [-1, 0, 1, 1, 7, 0, 0, 3]:
    #   row 0: -127 + 0 + 34 - 32 + 0 + 0 + 0 + 6 = -119   -> -119 / 64
    #   row 1: -1 + 0 + 2 + 4 + 0 + 0 + 0 + 0 = 5          -> 5 / 32
    xi = np.array([[1, 2, 0, -1, 3, 1, 5, -2], [-1, 0, 1, 1, 7, 0, 0, 3]], dtype=np.float32)
    y = oracle.q8_gemm_f64(wl.to_bf16_bits(xi), w)
    assert y.tolist() == [[92 / 64, -257 / 32], [-119 / 64, 5 / 32]]


def test_hand_worked_blob_with_escapes():
    """A 128 x 512 matrix (one tile, two segments) built so that its escapes
    can be listed by hand.  Each segment holds +0.0 almost everywhere and the
    fourteen exponents 100..113 twice each, so its table is {0, 100..113} and
    any other exponent escapes.  The escapes (value 2^(e-127), sign and
    mantissa 0) are placed so that the quarter -> chunk -> row -> column order
    differs from plain row-major order:
      segment 0: e=120 at (5, 3)    quarter 0, chunk 0
                 e=121 at (33, 40)  quarter 1, chunk 1
                 e=122 at (60, 5)   quarter 1, chunk 0
                 e=123 at (60, 1)   quarter 1, chunk 0
      segment 1: e=124 at (100, 300) quarter 3, chunk 1 of the segment
    so the escape plane reads 120, 123, 122, 121 | 124."""
    n, k = 128, 512
    w = np.zeros((n, k), dtype=np.uint16)
    for s in range(2):
        for i in range(14):
            col = 256 * s + 10 + i
            w[70 + i, col] = w[90 + i, col] = np.uint16((100 + i) << 7)
    for (r, c), e in {(5, 3): 120, (33, 40): 121, (60, 5): 122, (60, 1): 123, (100, 300): 124}.items():
        w[r, c] = np.uint16(e << 7)
    blob = oracle.encode(w)
    # geometry: 2 segment headers (64 B, plane padded to 256), 16 chunks
    assert _hdr(blob, 0x58, 8) == 256 and _hdr(blob, 0x60, 8) == 64
    assert _hdr(blob, 0x68, 8) == 512 and _hdr(blob, 0x70, 8) == 16 * 6144
    off_e = 512 + 16 * 6144
    assert _hdr(blob, 0x78, 8) == off_e and _hdr(blob, 0x80, 8) == 5 and _hdr(blob, 0x88, 8) == 16
    assert _hdr(blob, 0x90, 8) == blob.size == off_e + 256
    assert list(blob[off_e:off_e + 16]) == [120, 123, 122, 121, 124] + [0] * 11
    for s, (base, counts, mask) in enumerate([(0, [1, 3, 0, 0], 0x301), (4, [0, 0, 0, 1], 1 << 25)]):
        hd = blob[256 + 32 * s:256 + 32 * (s + 1)]
        assert sorted(int(v) for v in hd[:15]) == sorted([0] + list(range(100, 114))) and hd[15] == 0
        assert int.from_bytes(bytes(hd[16:20]), "little") == base
        assert [int.from_bytes(bytes(hd[20 + 2 * q:22 + 2 * q]), "little") for q in range(4)] == counts
        assert int.from_bytes(bytes(hd[28:32]), "little") == mask

    def code(r, c):
        chunk = blob[512 + 6144 * (c // 32):512 + 6144 * (c // 32 + 1)]
        byte = int(chunk[4096 + 16 * r + (c % 32) // 2])
        return (byte >> 4) if c % 2 else (byte & 15)

    for r, c in [(5, 3), (33, 40), (60, 5), (60, 1), (100, 300)]:
        assert code(r, c) == 15
    assert code(70, 10) != 15 and code(0, 0) != 15
    assert np.array_equal(oracle.decode(blob), w)
