"""Pins for the CPU oracle: each test checks it against something other than itself — closed
forms, exact rational arithmetic, brute force, library casts, invariants and the constants the
pages print — chosen so that a dropped term, a wrong sign, index or operand fails one of them.

Page references: "optimize the compressor 128 split cutedsl kernel" (vLLM PR #44230) and the
docs.vllm.ai API page of vllm.models.deepseek_v4.common.ops.fused_compress_quant_cache,
kernel _fused_kv_compress_norm_rope_insert_sparse_attn.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from deepseek_v4_sparse_c128_gb300 import inputs

GOLD = os.path.join(os.path.dirname(__file__), "golden")
CONST = {k: v["value"] for k, v in json.load(open(os.path.join(GOLD, "pages_constants.json"))).items()
         if not k.startswith("_")}
HEAD, NOPE, ROPE, QB = CONST["head_size"], CONST["nope_dim"], CONST["rope_dim"], CONST["quant_block"]
TS, SD = CONST["token_stride"], CONST["scale_dim"]
F32_MAX = float(np.finfo(np.float32).max)


# ----------------------------------------------------------------------------- exact helpers
def rn32_of_fraction(x: Fraction) -> np.float32:
    """Round an exact rational to binary32, nearest-even, by comparing against neighbours."""
    if x == 0:
        return np.float32(0.0)
    if x >= Fraction(F32_MAX) + Fraction(2) ** 103:
        return np.float32(np.inf)
    f = np.float32(float(x))
    cands = {f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))}
    cands = [c for c in cands if np.isfinite(c)]

    def key(c):
        return (abs(Fraction(float(c)) - x), int(np.array(c, np.float32).view(np.uint32)) & 1)
    return min(cands, key=key)


def e4m3_value(code: int) -> float:
    """Decode an e4m3fn byte from the format definition (bias 7, 3 mantissa bits)."""
    s = -1.0 if code & 0x80 else 1.0
    E, m = (code >> 3) & 15, code & 7
    if E == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1 + m / 8.0) * 2.0 ** (E - 7)


def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------------------------ pages
def test_constants_match_pages():
    """The oracle's layout and limits are the numbers the pages print."""
    assert HEAD == NOPE + ROPE == 512
    assert CONST["rows_per_window"] == CONST["compress_ratio"] == 128
    assert CONST["compress_ratio"] // CONST["state_block_size"] == 16
    assert NOPE // QB == CONST["nope_scale_bytes"] == SD - 1
    assert TS == NOPE + 2 * ROPE
    assert oracle.TOKEN_STRIDE == TS and oracle.SCALE_DIM == SD and oracle.HEAD == HEAD
    # largest e4m3 magnitude is FP8_MAX, and it is what saturation gives
    assert e4m3_value(oracle.e4m3_code(CONST["fp8_max"])) == CONST["fp8_max"]
    assert oracle.e4m3_code(1e9) == 0x7E
    # the absmax floor: an all-zero vector gets scale byte bias + ceil(log2(RN32(1e-4)*RN32(1/448)))
    tok, sc = oracle.epilogue(np.zeros(512, np.float32), np.ones(512, np.float32), 1e-6,
                              np.zeros(64, np.float32))
    raw = Fraction(float(np.float32(CONST["absmax_floor"]))) * Fraction(float(np.float32(1 / 448)))
    e = math.ceil(math.log2(float(raw)))
    assert Fraction(2) ** e >= raw > Fraction(2) ** (e - 1)
    assert list(sc) == [CONST["ue8m0_bias"] + e] * 7 + [0]
    assert not tok.any()


# ------------------------------------------------------------------------------- encoders
def test_bf16_encoder_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    u = u[((u >> 23) & 0xFF) != 0xFF]                        # finite patterns only
    ties = (rng.integers(0, 2 ** 16, size=50_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties[((ties >> 23) & 0xFF) != 0xFF]
    x = np.concatenate([u, ties, np.array([0x7F7FFFFF, 0xFF7FFFFF, 0, 0x80000000, 1, 0x807FFFFF], np.uint32)])
    x = x.view(np.float32)
    ours = oracle.bf16_bits_array(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def _e4m3_probe_values():
    rng = np.random.default_rng(12)
    mags = np.array(sorted({abs(e4m3_value(c)) for c in range(127)}), np.float64)
    mids = (mags[:-1] + mags[1:]) / 2                         # exact ties (representable in fp32)
    mids32 = mids.astype(np.float32)
    assert np.array_equal(mids32.astype(np.float64), mids)
    near = np.concatenate([np.nextafter(mids32, np.float32(0)), np.nextafter(mids32, np.float32(1e9))])
    bf = (np.arange(2 ** 16, dtype=np.uint32) << 16).view(np.float32)   # every bf16 value
    bf = bf[np.isfinite(bf) & (np.abs(bf) <= 448)]
    rnd = (rng.random(200_000) * 2 - 1) * 448 * 2.0 ** -rng.integers(0, 40, size=200_000)
    vals = np.concatenate([mids32, near, bf, rnd.astype(np.float32), mags.astype(np.float32)])
    return np.concatenate([vals, -vals]).astype(np.float32)


def test_e4m3_encoder_matches_torch_cast():
    """Nearest-even e4m3fn encoding of |y| <= 448 (the clamp keeps the op there)."""
    torch = pytest.importorskip("torch")
    x = _e4m3_probe_values()
    ours = oracle.e4m3_codes(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(ours[i]), int(ref[i])) for i in bad[:10]]


def test_e4m3_encoder_definition():
    """Decode(encode(v)) == v for every finite code; the sign of zero and of underflow is kept."""
    for c in list(range(0, 127)) + list(range(128, 255)):
        v = e4m3_value(c)
        if c == 0x80:
            continue
        assert oracle.e4m3_code(v) == c, c
    assert oracle.e4m3_code(-0.0) == 0x80
    assert oracle.e4m3_code(-1e-30) == 0x80
    assert oracle.e4m3_code(2.0 ** -10) == 0x00          # tie between 0 and 2^-9: even code
    assert oracle.e4m3_code(3 * 2.0 ** -10) == 0x02      # tie between 2^-9 (01) and 2^-8 (02)
    assert oracle.e4m3_code(464.0 - 1e-3) == 0x7E and oracle.e4m3_code(-1000.0) == 0xFE


def test_ceil_log2_brute_force():
    rng = np.random.default_rng(13)
    xs = np.exp(rng.uniform(math.log(1e-30), math.log(1e30), 20_000)).astype(np.float32)
    pw = np.float32(2.0) ** np.arange(-126, 127, dtype=np.float32)
    xs = np.concatenate([xs, pw, np.nextafter(pw, np.float32(0)), np.nextafter(pw, np.float32(np.inf))])
    for x in xs:
        xv = float(x)
        e = -160
        while math.ldexp(1.0, e) < xv:
            e += 1
        assert oracle.ceil_log2(x) == e, xv


# ----------------------------------------------------------------------------- variance
def _exact_mean_square(c: np.ndarray) -> np.float32:
    s = sum((Fraction(float(v)) ** 2 for v in c), Fraction(0))
    return rn32_of_fraction(s / 512)


@pytest.mark.parametrize("case", range(14))
def test_mean_square_is_exact_rounding(case):
    rng = np.random.default_rng(100 + case)
    c = np.zeros(512, np.float32)
    if case == 0:
        c = rng.standard_normal(512).astype(np.float32)
    elif case == 1:
        c = (rng.standard_normal(512) * 1e-20).astype(np.float32)
    elif case == 2:
        c = (rng.standard_normal(512) * 1e15).astype(np.float32)
    elif case == 3:    # magnitudes spread over 2^-60 .. 2^60
        c = (rng.standard_normal(512) * 2.0 ** rng.integers(-60, 61, 512)).astype(np.float32)
    elif case == 4:    # subnormal inputs, subnormal result
        c = (rng.standard_normal(512) * 1e-41).astype(np.float32)
    elif case == 5:    # exact tie: 1 + 2^-24 -> ties to even (down)
        c[0], c[1] = 1.0, 2.0 ** -12
    elif case == 6:    # just above the tie -> up
        c[0], c[1], c[2] = 1.0, 2.0 ** -12, 2.0 ** -40
    elif case == 7:    # 1 + 3*2^-24 is a tie with an odd lower neighbour -> up
        c[0], c[1:4] = 1.0, 2.0 ** -12
    elif case == 8:    # overflow to +inf
        c[:] = 2.0 ** 70
    elif case == 9:    # all zero
        pass
    elif case == 10:   # one huge and many tiny: the tiny ones still decide the rounding
        c[0] = 1.0
        c[1:] = np.float32(2.0 ** -30)
    elif case == 11:   # a sum that naive fp32 accumulation in index order gets wrong
        c = np.random.default_rng(0).standard_normal(512).astype(np.float32)
    elif case == 12:
        c = rng.uniform(-3, 3, 512).astype(np.float32)
    elif case == 13:   # the smallest subnormal
        c[:7] = np.float32(1e-45)
    got = oracle.mean_square_512(c)
    want = _exact_mean_square(c)
    assert got.view(np.uint32) == want.view(np.uint32), (got, want)
    if case == 11:
        naive = np.float32(0)
        for v in c:
            naive = np.float32(naive + np.float32(v * v))
        assert np.float32(naive / np.float32(512)) != want     # the case discriminates


# ----------------------------------------------------------------------------- epilogue
def _hand_code(v: float) -> int:
    """e4m3 code of v = +-(1 + f) * 2^j written out from the format (f in eighths, or ties)."""
    s = 0x80 if v < 0 or (v == 0 and math.copysign(1, v) < 0) else 0
    a = abs(v)
    if a == 0:
        return s
    j = math.floor(math.log2(a))
    frac = a / 2.0 ** j - 1.0                      # in [0, 1)
    if j < -6:                                     # subnormal range: multiples of 2^-9
        m = a / 2.0 ** -9
        lo = math.floor(m)
        m = lo + (1 if (m - lo > 0.5 or (m - lo == 0.5 and lo % 2 == 1)) else 0)
        return s | int(m) if m < 8 else s | (1 << 3)
    e8 = frac * 8
    lo = math.floor(e8)
    m = lo + (1 if (e8 - lo > 0.5 or (e8 - lo == 0.5 and lo % 2 == 1)) else 0)
    if m == 8:
        j, m = j + 1, 0
    return s | ((j + 7) << 3) | m


def _closed_form_case(rng):
    """comp in {0, +-1, +-2} with mean square exactly 1 (rrms = 1 when eps = 0); rms_w picks
    exact per-column values so normed = comp * w is known exactly."""
    comp = np.zeros(512, np.float32)
    for g in range(128):
        if rng.random() < 0.5:
            comp[4 * g:4 * g + 4] = rng.choice([-1.0, 1.0], 4)
        else:
            comp[4 * g + rng.integers(0, 4)] = rng.choice([-2.0, 2.0])
    assert float(np.sum(comp.astype(np.float64) ** 2)) == 512.0
    mant = np.array([1.0, 1.5, 1.0625, 1.1875, 1.25, 1.75])
    w = np.zeros(512, np.float32)
    for b in range(8):
        eb = int(rng.integers(-12, 4))                 # per-block magnitude, incl. e4m3 subnormals
        w[64 * b:64 * b + 64] = (rng.choice(mant, 64) * 2.0 ** (eb + rng.integers(-8, 1, 64))).astype(np.float32)
    return comp, w


def test_epilogue_closed_form():
    """RMSNorm with var = 1 and eps = 0, power-of-two scaling and exact FP8/bf16 codes by hand."""
    rng = np.random.default_rng(21)
    inv448 = Fraction(float(np.float32(1 / 448)))      # RN32(1/448), as the page's constexpr
    for _ in range(40):
        comp, w = _closed_form_case(rng)
        C, S = float(rng.choice([1.0, 0.0, 0.5, -1.0])), float(rng.choice([0.0, 1.0, 0.5, -0.5]))
        cs = np.concatenate([np.full(32, C, np.float32), np.full(32, S, np.float32)])
        tok, sc = oracle.epilogue(comp, w, 0.0, cs)
        normed = comp.astype(np.float64) * w.astype(np.float64)          # exact
        assert np.array_equal(normed.astype(np.float32).astype(np.float64), normed)
        for b in range(7):
            x = normed[64 * b:64 * b + 64]
            amax = max(float(np.max(np.abs(x))), float(np.float32(1e-4)))
            raw = Fraction(float(rn32_of_fraction(Fraction(amax) * inv448)))  # fp32 product
            e = math.ceil(math.log2(float(raw)))
            if Fraction(2) ** (e - 1) >= raw:
                e -= 1
            assert Fraction(2) ** e >= raw > Fraction(2) ** (e - 1)
            assert sc[b] == 127 + e
            want = [_hand_code(float(np.clip(v * 2.0 ** -e, -448, 448))) for v in x]
            assert list(tok[64 * b:64 * b + 64]) == want, b
        assert sc[7] == 0
        ev, od = normed[448::2], normed[449::2]
        ne, no = ev * C - od * S, od * C + ev * S                      # exact for these values
        got = tok[448:].view(np.uint16)
        want_e = oracle.bf16_bits_array(ne.astype(np.float32))
        want_o = oracle.bf16_bits_array(no.astype(np.float32))
        assert np.array_equal(ne.astype(np.float32).astype(np.float64), ne)
        assert np.array_equal(got[0::2], want_e) and np.array_equal(got[1::2], want_o)


def test_epilogue_rmsnorm_scaling():
    """rrms = 1/sqrt(var + eps): comp = +-2 gives normed +-1; comp = +-1 with eps = 3 gives
    normed +-0.5 (eps sits inside the root)."""
    rng = np.random.default_rng(22)
    signs = rng.choice([-1.0, 1.0], 512).astype(np.float32)
    ones = np.ones(512, np.float32)
    ident = np.concatenate([np.ones(32, np.float32), np.zeros(32, np.float32)])
    for comp, eps, mag, e in ((2 * signs, 0.0, 1.0, -8), (signs, 3.0, 0.5, -9)):
        tok, sc = oracle.epilogue(comp, ones, eps, ident)
        # amax = mag -> e = ceil(log2(mag/448)); y = +-mag*2^-e = +-256 -> code 0x78 / 0xF8
        assert list(sc) == [127 + e] * 7 + [0]
        assert np.array_equal(tok[:448], np.where(signs[:448] < 0, 0xF8, 0x78).astype(np.uint8))
        assert np.array_equal(bf16_to_f32(tok[448:].view(np.uint16)), mag * signs[448:])


def test_epilogue_random_properties():
    """Against an fp64 restatement with tolerances: block exponents, dequantised values,
    rotation (cos at [j], sin at [32+j], even/odd pairs) and pair norms."""
    rng = np.random.default_rng(23)
    for it in range(60):
        comp = (rng.standard_normal(512) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        w = (1 + 0.1 * rng.standard_normal(512)).astype(np.float32)
        eps = float(rng.choice([1e-6, 0.0, 1e-2]))
        ang = rng.uniform(0, 2 * np.pi, 32)
        cs = np.concatenate([np.cos(ang), np.sin(ang)]).astype(np.float32)
        tok, sc = oracle.epilogue(comp, w, eps, cs)
        c64 = comp.astype(np.float64)
        normed = c64 / np.sqrt(np.mean(c64 ** 2) + np.float32(eps)) * w
        for b in range(7):
            x = normed[64 * b:64 * b + 64]
            amax = np.max(np.abs(x))
            r = math.log2(max(amax, 1e-4) / 448)
            if abs(r - round(r)) > 4e-3:          # beyond what the bf16 pre-round can move
                assert sc[b] == 127 + math.ceil(r)
            scale = 2.0 ** (int(sc[b]) - 127)
            deq = np.array([e4m3_value(int(t)) for t in tok[64 * b:64 * b + 64]]) * scale
            err = np.abs(deq - x)
            assert np.all(err <= np.abs(x) * (2 ** -4 + 2 ** -8) + 2 ** -10 * scale * 1.01), (it, b)
        ev, od = normed[448::2], normed[449::2]
        C, S = cs[:32].astype(np.float64), cs[32:].astype(np.float64)
        ne, no = ev * C - od * S, od * C + ev * S
        got = bf16_to_f32(tok[448:].view(np.uint16)).astype(np.float64)
        tol = 2 ** -8 * (np.abs(ev) + np.abs(od)) + 1e-30
        assert np.all(np.abs(got[0::2] - ne) <= tol) and np.all(np.abs(got[1::2] - no) <= tol)
        assert np.allclose(np.hypot(got[0::2], got[1::2]), np.hypot(ev, od), rtol=2 ** -7)


# ---------------------------------------------------------------------- softmax / weighted sum
def _window(rng):
    rows = np.empty((128, 1024), np.float32)
    rows[:, :512] = rng.standard_normal((128, 512))
    rows[:, 512:] = 2 * rng.standard_normal((128, 512))
    return rows


def test_compress_constant_kv_is_exact():
    """Weights sum to one: kv constant down a column gives exactly that constant."""
    rng = np.random.default_rng(31)
    rows = _window(rng)
    k = rng.standard_normal(512).astype(np.float32)
    rows[:, :512] = k[None, :]
    assert np.array_equal(oracle.compress_rows(rows), k)


def test_compress_constant_score_is_mean():
    rng = np.random.default_rng(32)
    rows = _window(rng)
    rows[:, 512:] = rng.standard_normal(512).astype(np.float32)[None, :]
    want = rows[:, :512].astype(np.float64).mean(axis=0)
    got = oracle.compress_rows(rows).astype(np.float64)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2 ** -23 + 1e-300)


def test_compress_one_hot_selects_row():
    """Score 0 on one row and -200 elsewhere selects that row's kv exactly; rows are in order."""
    rng = np.random.default_rng(33)
    rows = _window(rng)
    pick = rng.integers(0, 128, 512)
    rows[:, 512:] = -200.0
    rows[pick, 512 + np.arange(512)] = 0.0
    assert np.array_equal(oracle.compress_rows(rows), rows[pick, np.arange(512)])


def test_compress_two_rows_closed_form():
    """Two live rows: comp = kv_b + (kv_a - kv_b) / (1 + e^(s_b - s_a)) (natural exp)."""
    rng = np.random.default_rng(34)
    rows = _window(rng)
    rows[:, 512:] = -1000.0
    a, b = 5, 77
    sa = rng.uniform(-3, 3, 512).astype(np.float32)
    sb = rng.uniform(-3, 3, 512).astype(np.float32)
    rows[a, 512:], rows[b, 512:] = sa, sb
    ka, kb = rows[a, :512].astype(np.float64), rows[b, :512].astype(np.float64)
    want = kb + (ka - kb) / (1.0 + np.exp(sb.astype(np.float64) - sa.astype(np.float64)))
    got = oracle.compress_rows(rows).astype(np.float64)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2 ** -23 + 1e-12)


def test_compress_invariances():
    """Shift of the scores and a permutation of the rows leave comp unchanged; scaling kv by 2
    scales comp by exactly 2."""
    rng = np.random.default_rng(35)
    rows = _window(rng)
    rows[:, 512:] = np.round(rows[:, 512:] * 2 ** 16) / 2 ** 16   # on a grid: +0.5 stays exact
    base = oracle.compress_rows(rows)
    shifted = rows.copy()
    shifted[:, 512:] += np.float32(0.5)
    perm = rows[rng.permutation(128)]
    doubled = rows.copy()
    doubled[:, :512] *= 2
    for other in (oracle.compress_rows(shifted), oracle.compress_rows(perm)):
        assert np.all(np.abs(other - base) <= np.spacing(np.abs(base)))   # at most one ulp
    assert np.array_equal(oracle.compress_rows(doubled), 2 * base)


# ------------------------------------------------------------------------------- whole op
def _single_token_problem(rng, pos, kv_slot, bs=2, nkb=4, nb=64, mb=64):
    p = inputs.random_problem(int(rng.integers(1 << 30)), 1, 1, mb, nb, bs)
    p.token_to_req[:] = 0
    p.positions[:] = pos
    p.slot_mapping[:] = 5
    p.kv_slot_mapping[:] = kv_slot
    p.block_table[0] = rng.permutation(nb)[:mb]
    p.k_cache = rng.integers(0, 256, size=(nkb, bs, 584), dtype=np.uint8)
    p.cos_sin = inputs._cos_sin_cache(mb * 8)
    return p


def test_gather_reads_the_window_rows():
    """Identity-coded state: kv = block*8 + row; a one-hot score picks window row i(c) = c % 128.
    comp[c] then names the physical row read, which must be block_table[(p-127+i)//8],
    offset (p-127+i)%8."""
    rng = np.random.default_rng(41)
    for pos in (127, 255, 1023, 4095, 511):
        p = _single_token_problem(rng, pos, kv_slot=3, nb=1024, mb=512)
        nb = p.state.shape[0]
        ident = (np.arange(nb)[:, None] * 8 + np.arange(8)[None, :]).astype(np.float32)
        p.state[..., :512] = ident[..., None]
        p.state[..., 512:] = -200.0
        start = pos - 127
        i_of_c = np.arange(512) % 128
        for c in range(512):
            q = start + i_of_c[c]
            p.state[p.block_table[0, q // 8], q % 8, 512 + c] = 0.0
        comp = np.zeros((1, 512), np.float32)
        oracle.forward(p, comp_out=comp)
        q = start + i_of_c
        want = p.block_table[0, q // 8].astype(np.float32) * 8 + q % 8
        assert np.array_equal(comp[0], want), pos


def test_store_layout_and_untouched_bytes():
    """kv slot s of a bs-slot cache: token bytes at blk*stride + off*576, scales at
    blk*stride + bs*576 + off*8, 7 exponents then a zero pad; every other byte unchanged."""
    rng = np.random.default_rng(42)
    for bs, slot in ((2, 3), (2, 0), (64, 77), (1, 2)):
        p = _single_token_problem(rng, 255, kv_slot=slot, bs=bs, nkb=4)
        kc = oracle.forward_k_cache(p)
        flat0, flat1 = p.k_cache.reshape(-1), kc.reshape(-1)
        stride = bs * 584
        blk, off = slot // bs, slot % bs
        tok = np.arange(blk * stride + off * 576, blk * stride + off * 576 + 576)
        scl = np.arange(blk * stride + bs * 576 + off * 8, blk * stride + bs * 576 + off * 8 + 8)
        mask = np.zeros(flat0.size, bool)
        mask[tok] = True
        mask[scl] = True
        assert np.array_equal(flat0[~mask], flat1[~mask])
        assert flat1[scl[7]] == 0 and np.all(flat1[scl[:7]] > 90)
        comp = np.zeros((1, 512), np.float32)
        oracle.forward(p, comp_out=comp)
        t2, s2 = oracle.epilogue(comp[0], p.rms_w, p.eps, p.cos_sin[128])
        assert np.array_equal(flat1[tok], t2) and np.array_equal(flat1[scl], s2)


def test_activity_predicate():
    """Only slot >= 0, p >= 0, (p+1) % 128 == 0 and kv slot >= 0 write; p = -1 does not."""
    p = inputs.random_problem(7, 64, 4, 64, 64, 2, active_frac=0.0, pad_frac=0.0, kv_drop_frac=0.0)
    p.positions[:] = 126
    p.positions[:6] = [127, -1, 255, 383, -129, 128]
    p.slot_mapping[:] = 9
    p.slot_mapping[2] = -1          # padded token at a window end
    p.kv_slot_mapping[3] = -1       # window end without a kv slot
    kc = oracle.forward_k_cache(p)
    stride = 2 * 584
    written = set()
    for t in range(p.num_tokens):
        s = int(p.kv_slot_mapping[t])
        lo = (s // 2) * stride + (s % 2) * 576
        if s >= 0 and not np.array_equal(kc.reshape(-1)[lo:lo + 576], p.k_cache.reshape(-1)[lo:lo + 576]):
            written.add(t)
    assert written == {0}
    assert (kc != p.k_cache).sum() > 500


def test_paging_invariance():
    """Moving physical blocks and rewriting the block table changes no output byte."""
    p = inputs.make_problem("tiny")
    kc_a = oracle.forward_k_cache(p)
    rng = np.random.default_rng(44)
    perm = rng.permutation(p.state.shape[0])          # new home of old block b is perm[b]
    st = np.empty_like(p.state)
    st[perm] = p.state
    p.state = st
    p.block_table = perm[p.block_table].astype(np.int32)
    kc_b = oracle.forward_k_cache(p)
    assert np.array_equal(kc_a, kc_b)


def test_out_of_range_indices_report_and_skip():
    rng = np.random.default_rng(45)
    cases = [("req", 1), ("bt_col", 2), ("block", 4), ("cos_row", 8), ("kv_slot", 16)]
    for what, bit in cases:
        p = _single_token_problem(rng, 255, kv_slot=1)
        if what == "req":
            p.token_to_req[:] = 1
        elif what == "bt_col":
            p.positions[:] = 64 * 8 + 127
            p.cos_sin = inputs._cos_sin_cache(2048)
        elif what == "block":
            p.block_table[0, 20] = p.state.shape[0]
        elif what == "cos_row":
            p.cos_sin = p.cos_sin[:100]
        elif what == "kv_slot":
            p.kv_slot_mapping[:] = 8
        kc = p.k_cache.copy()
        err = oracle.forward(p, k_cache=kc)
        assert err == bit, what
        assert np.array_equal(kc, p.k_cache)


def test_threads_and_subsets_agree():
    p = inputs.make_problem("decode")
    a = oracle.forward_k_cache(p)
    b = oracle.forward_k_cache(p, threads=4)
    assert np.array_equal(a, b)
    half = np.arange(0, p.num_tokens, 2)
    c = p.k_cache.copy()
    oracle.forward(p, k_cache=c, tokens=half)
    oracle.forward(p, k_cache=c, tokens=np.arange(1, p.num_tokens, 2))
    assert np.array_equal(a, c)


def test_golden_tiny_regression():
    """The oracle's bytes for the tiny workload, stored by tests/golden/make_golden.py."""
    g = json.load(open(os.path.join(GOLD, "tiny_oracle.json")))
    p = inputs.make_problem("tiny")
    kc = oracle.forward_k_cache(p)
    comp = np.zeros((p.num_tokens, 512), np.float32)
    oracle.forward(p, comp_out=comp)
    assert kc.tobytes().hex() == g["k_cache_hex"]
    assert comp.tobytes().hex() == g["comp32_hex"]


# ------------------------------------------------------------------------------ rsqrt step
def test_rsqrt_is_correctly_rounded_fraction():
    """The oracle's rrms step against exact rational arithmetic: y is correctly rounded iff the
    midpoints to its neighbours bracket 1/sqrt(v), i.e. md^2 v < 1 < mu^2 v."""
    rng = np.random.default_rng(51)
    u = rng.integers(1, 0x7F800000, size=20_000, dtype=np.uint64).astype(np.uint32)
    vals = np.concatenate([u.view(np.float32), np.float32([1.0, 2.0, 0.5, 1e-6, 3.0, 1e-45, 3.4e38])])
    for v in vals:
        y = oracle.rsqrt(v)
        up, dn = np.nextafter(y, np.float32(np.inf)), np.nextafter(y, np.float32(0))
        fv, fy = Fraction(float(v)), Fraction(float(y))
        mu, md = (fy + Fraction(float(up))) / 2, (fy + Fraction(float(dn))) / 2
        assert md * md * fv < 1 < mu * mu * fv, float(v)


def test_rsqrt_exhaustive_check_program():
    """Compile tests/rsqrt_exhaustive.c and run it over every 509th positive fp32 pattern (all of
    them when C128_EXHAUSTIVE=1: 2,139,095,039 values, about a minute on 8 cores)."""
    import subprocess
    import tempfile
    src = os.path.join(os.path.dirname(__file__), "rsqrt_exhaustive.c")
    exe = os.path.join(tempfile.mkdtemp(), "rsqrt_exhaustive")
    subprocess.check_call([os.environ.get("CC", "cc"), "-O2", "-ffp-contract=off", "-o", exe, src, "-lm"])
    full = os.environ.get("C128_EXHAUSTIVE") == "1"
    step = 1 if full else 509
    n = 8
    bounds = [1 + i * ((0x7F800000 - 1) // n) for i in range(n)] + [0x7F800000]
    procs = [subprocess.Popen([exe, str(bounds[i]), str(bounds[i + 1]), str(step)], stdout=subprocess.PIPE, text=True)
             for i in range(n)]
    total = 0
    for pr in procs:
        out, _ = pr.communicate()
        assert pr.returncode == 0, out
        total += int(out.split()[1])
    assert total >= (0x7F800000 - 1) // step - n


# ------------------------------------------------- other configurations of the fused kernels
E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_encoder_definition():
    """E2M1: every code round-trips; ties go to the even code; beyond 6 saturates; sign kept."""
    for c in range(16):
        v = E2M1_MAG[c & 7] * (-1 if c & 8 else 1)
        if c == 8:
            continue
        assert oracle.e2m1_code(v) == c, c
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in ties.items():
        assert oracle.e2m1_code(v) == c and oracle.e2m1_code(-v) == c | 8, v
    assert oracle.e2m1_code(0.26) == 1 and oracle.e2m1_code(5.01) == 7
    assert oracle.e2m1_code(7.0) == 7 and oracle.e2m1_code(1e9) == 7 and oracle.e2m1_code(-0.0) == 8
    assert oracle.e2m1_code(-1e-30) == 8


def test_mean_square_128_is_exact():
    rng = np.random.default_rng(61)
    for scale in (1.0, 1e-20, 1e18):
        c = (rng.standard_normal(128) * scale).astype(np.float32)
        want = rn32_of_fraction(sum((Fraction(float(v)) ** 2 for v in c), Fraction(0)) / 128)
        assert oracle.mean_square_128(c).view(np.uint32) == want.view(np.uint32)


def _pow2_signs(rng, n, mags):
    return (rng.choice(mags, n) * rng.choice([-1.0, 1.0], n)).astype(np.float32)


def test_indexer_fp8_epilogue_closed_form():
    """Head 128: RMSNorm (var 1, eps 0), RoPE of the last 32 pairs only (cos at [j], sin at
    [32+j]) BEFORE the quant, one absmax over all 128 values, fp32 scale 2^e stored LE."""
    rng = np.random.default_rng(62)
    for it in range(30):
        comp = rng.choice([-1.0, 1.0], 128).astype(np.float32)        # mean square exactly 1
        w = (rng.choice([1.0, 1.5, 1.25, 1.75], 128) * 2.0 ** rng.integers(-6, 3, 128)).astype(np.float32)
        C, S = float(rng.choice([1.0, 0.0, -1.0, 0.5])), float(rng.choice([0.0, 1.0, -0.5]))
        cs = np.concatenate([np.full(32, C, np.float32), np.full(32, S, np.float32)])
        tok, sc = oracle.epilogue_indexer(1, comp, w, 0.0, cs)
        normed = comp.astype(np.float64) * w
        ev, od = normed[0::2].copy(), normed[1::2].copy()
        ne, no = ev.copy(), od.copy()
        ne[32:], no[32:] = ev[32:] * C - od[32:] * S, od[32:] * C + ev[32:] * S
        x = np.empty(128)
        x[0::2], x[1::2] = ne, no
        assert np.array_equal(x.astype(np.float32).astype(np.float64), x)    # exact so far
        x = bf16_to_f32(oracle.bf16_bits_array(x.astype(np.float32))).astype(np.float64)
        amax = max(float(np.abs(x).max()), float(np.float32(1e-4)))
        raw = Fraction(float(rn32_of_fraction(Fraction(amax) * Fraction(float(np.float32(1 / 448))))))
        e = math.ceil(math.log2(float(raw)))
        if Fraction(2) ** (e - 1) >= raw:
            e -= 1
        assert list(tok) == [_hand_code(float(np.clip(v * 2.0 ** -e, -448, 448))) for v in x]
        assert sc.view(np.float32)[0] == np.float32(2.0 ** e)


def test_indexer_mxfp4_epilogue_closed_form():
    """MXFP4: per 32 values amax -> e = ceil(log2(amax/6)), E2M1 codes of x*2^-e, byte j = even
    code | odd code << 4, UE8M0 byte e + 127; values chosen E2M1-exact at each block's scale."""
    rng = np.random.default_rng(63)
    inv6 = Fraction(float(np.float32(1 / 6)))
    for it in range(30):
        comp = rng.choice([-1.0, 1.0], 128).astype(np.float32)
        w = np.zeros(128, np.float32)
        ks = rng.integers(-10, 6, 4)
        for b in range(4):
            m = rng.choice([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], 32)
            m[rng.integers(0, 32)] = 6.0                                  # block max exactly 6 * 2^k
            w[32 * b:32 * b + 32] = (m * 2.0 ** ks[b]).astype(np.float32)
        cs = np.concatenate([np.ones(32, np.float32), np.zeros(32, np.float32)])  # rope = identity
        tok, sc = oracle.epilogue_indexer(2, comp, w, 0.0, cs)
        x = comp.astype(np.float64) * w
        for b in range(4):
            xb = x[32 * b:32 * b + 32]
            amax = float(np.abs(xb).max())
            ratio = Fraction(float(rn32_of_fraction(Fraction(amax) * inv6)))
            e = math.ceil(math.log2(float(ratio)))
            if Fraction(2) ** (e - 1) >= ratio:
                e -= 1
            assert e == ks[b] and sc[b] == e + 127
            codes = [E2M1_MAG.index(abs(v) * 2.0 ** -e) | (8 if v < 0 else 0) for v in xb]
            want = [codes[2 * j] | (codes[2 * j + 1] << 4) for j in range(16)]
            assert list(tok[16 * b:16 * b + 16]) == want, b


def test_forward_ex_matches_c128_forward():
    """The generic op with the C128 configuration is the C128 op, byte for byte."""
    p = inputs.make_problem("decode")
    a = oracle.forward_k_cache(p)
    b = p.k_cache.copy()
    assert oracle.forward_ex(p, k_cache=b) == 0
    assert np.array_equal(a, b)


def test_overlap_gather_and_masking():
    """Ratio 4 with overlap: 8 rows p-7..p; the older 4 read kv[0:H], score[SW:SW+H], the newer 4
    read kv[H:2H], score[SW+H:SW+2H]; rows at negative positions take no weight. Identity-coded
    kv + one-hot scores name the (block, row, half) each column read."""
    for fmt, head in ((0, 512), (1, 128)):
        p = inputs.prefill_problem("t", 3, 2, 12, 40, head, 4, 1, fmt)
        sw = p.state_width
        nb = p.state.shape[0]
        code = (np.arange(nb)[:, None] * 8 + np.arange(8)[None, :]).astype(np.float32)
        p.state[..., :sw] = code[..., None]
        p.state[..., head:2 * head] += np.float32(0.5)            # marks the newer half
        p.state[..., sw:] = -1000.0
        rng = np.random.default_rng(fmt)
        picks = {}
        for t in range(p.num_tokens):
            pos = int(p.positions[t])
            if (pos + 1) % 4 or p.kv_slot_mapping[t] < 0:
                continue
            r = int(p.token_to_req[t])
            valid = [i for i in range(8) if pos - 7 + i >= 0]
            pick = rng.choice(valid, head)
            picks[t] = pick
            for c in range(head):
                q = pos - 7 + pick[c]
                ho = head if pick[c] >= 4 else 0
                p.state[p.block_table[r, q // 8], q % 8, sw + ho + c] = 0.0
        # windows share rows (overlap), so check one token at a time on a fresh copy of the scores
        for t, pick in list(picks.items())[:12]:
            q2 = p.state.copy()
            pos, r = int(p.positions[t]), int(p.token_to_req[t])
            q2[..., sw:] = -1000.0
            for c in range(head):
                q = pos - 7 + pick[c]
                ho = head if pick[c] >= 4 else 0
                q2[p.block_table[r, q // 8], q % 8, sw + ho + c] = 0.0
            sub = inputs.Problem("x", p.token_to_req, p.positions, p.slot_mapping, p.block_table, q2, p.rms_w, p.eps,
                                 p.cos_sin, p.k_cache, p.kv_slot_mapping, p.kv_block_size, head=head, ratio=4,
                                 overlap=1, state_width=sw, fmt=fmt)
            comp = np.zeros((p.num_tokens, head), np.float32)
            oracle.forward_ex(sub, comp_out=comp, tokens=[t])
            q = pos - 7 + pick
            want = p.block_table[r, q // 8].astype(np.float32) * 8 + q % 8 + np.where(pick >= 4, 0.5, 0.0)
            assert np.array_equal(comp[t], want.astype(np.float32)), t


def test_indexer_absmax_floors():
    """The absmax floors of the indexer formats, in closed form. MXFP4: a block whose values are
    all zero has amax floored to 6*2^-126, RN32(6*2^-126 * RN32(1/6)) is exactly 2^-126 (the
    product is 2^-126 (1 + 3e-8), below half an ulp), so e = -126, the UE8M0 byte is 1, and every
    code is a zero (nibble 0 or 8, the sign of the zero). FP8 indexer: an all-zero vector has amax
    floored to RN32(1e-4), and the scale is 2^e with e = ceil(log2(RN32(RN32(1e-4) RN32(1/448))))."""
    rng = np.random.default_rng(64)
    comp = rng.choice([-1.0, 1.0], 128).astype(np.float32)
    w = rng.choice([0.5, 1.0, 2.0], 128).astype(np.float32)
    w[32:64] = 0.0                                                    # block 1 is all zeros
    cs = np.concatenate([np.ones(32, np.float32), np.zeros(32, np.float32)])
    tok, sc = oracle.epilogue_indexer(2, comp, w, 0.0, cs)
    assert sc[1] == 1
    for byte in tok[16:32]:
        assert (byte & 0xF) in (0, 8) and (byte >> 4) in (0, 8)
    assert all(s != 1 for b, s in enumerate(sc) if b != 1)
    # FP8 indexer, every value zero
    tok8, sc8 = oracle.epilogue_indexer(1, comp, np.zeros(128, np.float32), 1e-6, cs)
    floor = Fraction(float(np.float32(1e-4)))
    raw = Fraction(float(rn32_of_fraction(floor * Fraction(float(np.float32(1 / 448))))))
    e = math.ceil(math.log2(float(raw)))
    if Fraction(2) ** (e - 1) >= raw:
        e -= 1
    assert sc8.view(np.float32)[0] == np.float32(2.0 ** e)
    assert all(b in (0x00, 0x80) for b in tok8)
