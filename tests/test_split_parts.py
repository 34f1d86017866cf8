"""The bf16 part splits that let fp32 operands through bf16 tensor-core MMAs,
checked on the CPU with an emulation of round-to-nearest-even bf16:

* router weight, three parts: W0 = rn(W), W1 = rn(W - W0), W2 = rn(W - W0 - W1)
  (both differences exact in fp32), and W0 + W1 + W2 == W exactly for normal
  fp32 values -- the products with bf16 x are then exact and the logits keep
  fp32 accuracy;
* router-gradient operands, two parts: hi = rn(v), lo = rn(v - hi), with
  |v - hi - lo| <= 2^-16 |v|: for v in [2^e, 2^(e+1)), |v - hi| <= 2^(e-8) (half
  a bf16 ulp) and lo's rounding loses at most 2^(e-16); the worst case seen
  on the samples is ~2^-17.
"""
import numpy as np


def rn_bf16(v: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), returned as fp32."""
    u = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _samples(n=400_000, seed=3):
    g = np.random.default_rng(seed)
    mant = g.uniform(1.0, 2.0, n)
    expo = g.integers(-100, 100, n)
    sign = g.choice([-1.0, 1.0], n)
    v = (sign * mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    edge = np.array([1.0, -1.0, 1.0 + 2 ** -23, 1.0 - 2 ** -24, 3.0, 0.1, -0.02, 65504.0, 2 ** -100,
                     np.float32(1.0000001), np.float32(0.33333334)], dtype=np.float32)
    return np.concatenate([v, edge])


def test_emulated_rounding_matches_known_values():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9, 1.0 + 2 ** -9 + 2 ** -20], dtype=np.float32)
    # 8 significant bits (ulp 2^-7 on [1, 2)); 1 + 2^-8 is a tie and goes to the even neighbour 1.0
    want = np.array([1.0, 1.0, 1.0, 1.0 + 2 ** -7, 1.0], dtype=np.float32)
    assert np.array_equal(rn_bf16(x), want)


def test_three_part_router_weight_split_is_exact():
    w = _samples()
    w0 = rn_bf16(w)
    r1 = (w - w0).astype(np.float32)
    assert np.array_equal(r1.astype(np.float64), w.astype(np.float64) - w0.astype(np.float64))   # exact
    w1 = rn_bf16(r1)
    r2 = (r1 - w1).astype(np.float32)
    assert np.array_equal(r2.astype(np.float64), r1.astype(np.float64) - w1.astype(np.float64))  # exact
    w2 = rn_bf16(r2)
    total = w0.astype(np.float64) + w1.astype(np.float64) + w2.astype(np.float64)
    assert np.array_equal(total, w.astype(np.float64))


def test_two_part_split_error_bound():
    v = _samples(seed=5)
    hi = rn_bf16(v)
    lo = rn_bf16((v - hi).astype(np.float32))
    err = np.abs(v.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert np.all(err <= 2.0 ** -16 * np.abs(v.astype(np.float64)))
