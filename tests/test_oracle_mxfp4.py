"""Pins for the MXFP4 oracle against things other than itself (CPU only).

* E2M1 decode vs. IEEE half precision: the E2M1 bit fields placed into a
  float16 (e1 e0 m -> exponent bits 11..10 and mantissa bit 9, sign bit 15)
  give the E2M1 value times 2^-14, because E2M1's exponent-0 codes line up
  with float16 subnormals. numpy decodes the float16.
* E8M0 decode vs. torch's float8_e8m0fnu conversion.
* Rounding vs. the FPU's own round-to-nearest-even (np.rint) applied at the
  E2M1 grid spacing of each binade, then saturation at 6.
* The OCP scale rule's defining property: amax / X lies in [4, 8).
* Value idempotence of quantise(dequantise(.)).
Each pin also runs against planted mistakes to show it would catch them.
"""
import numpy as np
import pytest
import torch

from oracle import mxfp4


def f16_e2m1(codes):
    c = np.asarray(codes, dtype=np.uint16)
    bits = ((c & 7) << 9) | ((c & 8) << 12)
    return bits.view(np.float16).astype(np.float64) * 2.0 ** 14


def torch_e8m0(s):
    t = torch.tensor(np.asarray(s, dtype=np.uint8)).view(torch.float8_e8m0fnu)
    return t.to(torch.float64).numpy()


def rne_e2m1_reference(q):
    """Nearest E2M1 value by the FPU's RNE at the binade's grid spacing."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.rint(a / step) * step          # np.rint: round half to even
    r = np.minimum(r, 6.0)
    return np.where(np.signbit(q), -r, r)


# ---- pin checks (return True when the oracle agrees) -------------------------

def pin_decode(mod) -> bool:
    codes = np.arange(16)
    if not np.array_equal(mod.e2m1_decode(codes), f16_e2m1(codes)):
        return False
    s = np.arange(255)
    if not np.array_equal(mod.e8m0_decode(s), torch_e8m0(s)):
        return False
    # exhaustive code x scale through the packed interface
    cc, ss = np.meshgrid(np.arange(16), np.arange(255), indexing="ij")
    cc, ss = cc.ravel(), ss.ravel()
    n = cc.size                                  # 4080 = 127.5 blocks -> pad to 128 blocks
    pad = 128 * 32 - n
    codes_full = np.concatenate([cc, np.zeros(pad, dtype=np.int64)])
    # put one (code, scale) per block position: block b uses scale ss[...]
    # easiest: one element per row, rows of 32 with a single nonzero element
    rows = np.zeros((n, 32), dtype=np.uint8)
    rows[:, 0] = cc
    packed = mxfp4.pack_nibbles(rows)
    vals = mod.dequantize(packed, ss.astype(np.uint8)[:, None])
    want = f16_e2m1(cc) * torch_e8m0(ss)
    del codes_full
    return np.array_equal(vals[:, 0], want) and np.all(vals[:, 1:] == 0)


def pin_rounding(mod) -> bool:
    rng = np.random.default_rng(1)
    q = np.concatenate([rng.uniform(-7.99, 7.99, 20000), rng.uniform(-1, 1, 5000)])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    ulp = np.spacing(mids)
    probes = np.concatenate([mids, mids - ulp, mids + ulp, [0.0, 6.0, 7.0, 7.999, 0.5, 4.0]])
    q = np.concatenate([q, probes, -probes])
    got = mod.e2m1_decode(mod.round_to_e2m1(q))
    want = rne_e2m1_reference(q)
    # compare including the sign of zero (small negatives -> -0)
    return np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))


def pin_scale_rule(mod) -> bool:
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((64, 32 * 8)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    _, s, _ = mod.quantize(w)
    amax = np.abs(w.astype(np.float64)).reshape(64, 8, 32).max(-1)
    ratio = amax / np.ldexp(1.0, s.astype(np.int64) - 127)
    if not np.all((ratio >= 4.0) & (ratio < 8.0)):
        return False
    z = np.zeros((1, 32), dtype=np.float32)
    tiny = np.full((1, 32), 1e-40, dtype=np.float32)        # subnormal fp32 -> clamped to s = 0
    return mod.quantize(z)[1][0, 0] == 0 and mod.quantize(tiny)[1][0, 0] == 0


def pin_idempotent(mod) -> bool:
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, (50, 64))
    scales = rng.integers(100, 150, (50, 2)).astype(np.uint8)
    v = mod.dequantize(mxfp4.pack_nibbles(codes), scales)
    v2 = mod.fake_quantize(v.astype(np.float32))
    return np.array_equal(v, v2)


PINS = [pin_decode, pin_rounding, pin_scale_rule, pin_idempotent]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    assert pin(mxfp4)


def test_value_set_matches_format_definition():
    # OCP MX v1.0, FP4 E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
    assert list(mxfp4.e2m1_decode(range(8))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert list(mxfp4.e2m1_decode(range(8, 16))) == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert np.isnan(mxfp4.e8m0_decode(255))


def test_nibble_order_and_sign_of_zero():
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 0] = 6.0       # element 0 -> low nibble of byte 0
    w[0, 3] = -1e-9     # tiny negative -> -0 code 8, high nibble of byte 1
    c, s, _ = mxfp4.quantize(w)
    assert s[0, 0] == 127                          # 6 = 1.5 * 2^2, X = 2^0
    assert c[0, 0] == 0x07 and c[0, 1] == 0x80


def test_nonfinite_block_gets_nan_scale():
    w = np.ones((2, 64), dtype=np.float32)
    w[1, 40] = np.nan
    c, s, bad = mxfp4.quantize(w)
    assert bad and s[1, 1] == 255 and s[1, 0] != 255 and s[0, 1] != 255


def test_saturation():
    w = np.zeros((1, 32), dtype=np.float32)
    w[0, :2] = [7.5, 4.0]      # amax 7.5 -> X = 1, 7.5 saturates to 6
    c, s, _ = mxfp4.quantize(w)
    v = mxfp4.dequantize(c, s)
    assert v[0, 0] == 6.0 and v[0, 1] == 4.0


# ---- planted mistakes: each must fail at least one pin -----------------------

class _Mutant:
    def __init__(self, **over):
        self.__dict__.update({k: getattr(mxfp4, k) for k in dir(mxfp4) if not k.startswith("__")})
        self.__dict__.update(over)


def _mut_swapped_table():
    tbl = mxfp4.E2M1_MAGNITUDE.copy()
    tbl[[5, 6]] = tbl[[6, 5]]

    def dec(codes):
        c = np.asarray(codes, dtype=np.int64)
        m = tbl[c & 7]
        return np.where(c & 8, -m, m)
    m = _Mutant(e2m1_decode=dec)
    m.dequantize = lambda cp, s: dec(mxfp4.unpack_nibbles(cp)) * np.repeat(mxfp4.e8m0_decode(s), 32, -1)
    return m


def _mut_scale_bias():
    dec = lambda s: np.ldexp(1.0, np.asarray(s, dtype=np.int64) - 126)
    m = _Mutant(e8m0_decode=dec)
    m.dequantize = lambda cp, s: mxfp4.e2m1_decode(mxfp4.unpack_nibbles(cp)) * np.repeat(dec(s), 32, -1)
    return m


def _mut_ties_away():
    def rnd(q):
        q = np.asarray(q, dtype=np.float64)
        a = np.abs(q)
        d = np.abs(a[..., None] - mxfp4.E2M1_MAGNITUDE)
        best = d.min(-1, keepdims=True)
        mag = 7 - np.argmax((d == best)[..., ::-1], axis=-1)      # last (larger) of ties
        mag = np.where(a > 6, 7, mag)
        return (mag | (np.signbit(q).astype(np.int64) << 3)).astype(np.uint8)
    return _Mutant(round_to_e2m1=rnd)


def _mut_emax3():
    def se(amax):
        _, e = np.frexp(np.asarray(amax, dtype=np.float64))
        return np.where(np.asarray(amax) == 0, 0, np.clip(e - 1 - 3 + 127, 0, 254))

    def q(w):
        w = np.asarray(w, dtype=np.float32)
        K = w.shape[-1]
        v = w.astype(np.float64).reshape(*w.shape[:-1], K // 32, 32)
        s = se(np.abs(v).max(-1))
        codes = mxfp4.round_to_e2m1(v / np.ldexp(1.0, s - 127)[..., None]).reshape(w.shape)
        return mxfp4.pack_nibbles(codes), s.astype(np.uint8), False
    m = _Mutant(quantize=q)
    m.fake_quantize = lambda w: mxfp4.dequantize(*q(w)[:2])
    return m


def _mut_nibble_swap():
    def unpack(b):
        b = np.asarray(b, dtype=np.uint8)
        return np.stack([b >> 4, b & 0xF], -1).reshape(*b.shape[:-1], b.shape[-1] * 2)
    m = _Mutant()
    m.dequantize = lambda cp, s: mxfp4.e2m1_decode(unpack(cp)) * np.repeat(mxfp4.e8m0_decode(s), 32, -1)
    return m


@pytest.mark.parametrize("make", [_mut_swapped_table, _mut_scale_bias, _mut_ties_away,
                                  _mut_emax3, _mut_nibble_swap], ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(make):
    mutant = make()
    results = [pin(mutant) for pin in PINS]
    assert not all(results), "a planted mistake passed every pin"


def test_bf16_rounding_helper_matches_torch():
    """The parity tests' bf16 rounding (fp64 -> nearest bf16, ties to even)
    agrees with torch's fp32 -> bf16 conversion on fp32 inputs, including
    exact ties and values next to them."""
    import torch
    import oracle_par
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000))).astype(np.float32)
    bits = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F808001, 0x3F807FFF, 0x00008000, 0x7F7E8000],
                    dtype=np.uint32).view(np.float32)   # ties at even / odd mantissas, neighbours, subnormal, large (below the bf16 maximum)
    v = np.concatenate([v, bits])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_par.bf16_rne(v.astype(np.float64))
    assert np.array_equal(got, ref)
